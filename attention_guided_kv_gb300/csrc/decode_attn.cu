// Score-emitting split-K paged GQA decode attention (sm_103a).
//
// What it computes ("From sliding window to attention-guided eviction" §3.1
// and §4.2 step 1; "Long context, KV eviction and sparse attention",
// sparse-selection section): for each sequence and q head, softmax of the
// scaled logits against every live key, the weighted sum of V, every key's
// probability, and the H2O running score cum[kv head][key] += sum of the
// group's probabilities.
//
// Kernel 1 (decode_partial_kernel), grid (splits, Hkv, B), 5 warps:
//   * warp 4 lane 0 is the producer: it walks this split's pages through the
//     block table and TMA-loads each page's K and V rows of this kv head
//     (2 x 2 KB boxes each, 128-byte swizzle) into an 8-stage ring, with an
//     evict-first L2 policy (every byte is read once per step);
//   * warps 0..3 consume pages round-robin: S = Q K^T with mma.sync m16n8k16
//     (A = the group's q rows, at most 8 real rows; B = 16 keys via
//     ldmatrix), online softmax in the log2 domain, the raw log2-domain
//     logits written to the probability buffer, then O += P V where P is
//     split into a bf16 high part (rows 0..7 of A) and its bf16 residual
//     (rows 8..15), so P keeps ~16 mantissa bits at no extra MMA cost;
//   * the CTA merges its 4 warps and writes (m, l, unnormalised O) partials.
//   The CTA that owns the page of the appended slot first writes k_new /
//   v_new into the pool (and the slot's original position), then fences the
//   generic-proxy stores against its own later TMA reads.
// Kernel 2 (decode_finalize_kernel), grid (chunks, Hkv, B): merges the
//   split partials into O, rescales the stored logits into probabilities
//   exp2(s - M) / L in place, adds the group's sum into the H2O score and
//   publishes the new sequence length.
#include "common.cuh"

namespace kvsel {

constexpr int kD = 128;           // head_dim
constexpr int kPage = 16;         // tokens per page
constexpr int kStages = 8;        // TMA ring depth (pages)
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = 8192; // K (2 x 2 KB swizzled halves) + V (same)
constexpr int kMaxG = 8;
constexpr int kMaxSplits = 64;
constexpr int kFinalizeChunk = 2048;
constexpr size_t kPartialSmem = size_t(kStages) * kStageBytes + 1024 + 2 * kStages * 8;

struct DecodeParams {
  const int32_t* block_table;
  const int32_t* seq_lens;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  int32_t* pos_map;
  const int32_t* next_pos;
  float* logits;      // log2-domain logits [B][Hq][max_len] (probs buffer or workspace), or null
  float* part_ml;     // [B][Hkv][splits][G][2]
  float* part_o;      // [B][Hkv][splits][G][kD]
  int32_t* ws_len;    // [B] length after the append
  int* status;
  int max_pages, Hq, Hkv, G, num_pages, max_len, splits;
  float scale_log2;
};

// byte offset of 16-byte unit u (0..15, i.e. d = 8u..8u+7) of row `key` in a
// K or V page tile: two 64-column halves, each 16 rows x 128 B, swizzled by
// the TMA 128-byte pattern (unit ^= row & 7).
__device__ __forceinline__ uint32_t tile_off(int key, int u) {
  return (u >> 3) * 2048 + key * 128 + ((((u & 7) ^ (key & 7))) << 4);
}

__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int k0, int valid) {
  return v & ((k0 < valid ? 0x0000FFFFu : 0u) | (k0 + 1 < valid ? 0xFFFF0000u : 0u));
}

__global__ void __launch_bounds__(kThreads, 2)
decode_partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S_old = P.seq_lens[b];
  const bool append = P.k_new != nullptr;
  const int S = S_old + (append ? 1 : 0);
  const int npages = (S + kPage - 1) / kPage;
  const int pb = int((long long)split * npages / P.splits);
  const int pe = int((long long)(split + 1) * npages / P.splits);
  const int n = pe - pb;
  if (split == 0 && kvh == 0 && threadIdx.x == 0) P.ws_len[b] = S;
  if (S_old < 0 || S > P.max_len || npages > P.max_pages) {  // uniform per CTA
    if (threadIdx.x == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_fence_init();
  }
  if (threadIdx.x == kConsumerWarps * 32) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }

  // Append the new token (its page is loaded later by this CTA's producer).
  if (append) {
    const int ap = S_old / kPage;
    if (ap >= pb && ap < pe && threadIdx.x < 32) {
      const int phys = P.block_table[size_t(b) * P.max_pages + ap];
      if (unsigned(phys) < unsigned(P.num_pages)) {
        const size_t row = (size_t(phys) * P.Hkv + kvh) * kPage + (S_old % kPage);
        const int t = threadIdx.x & 15;
        const __nv_bfloat16* src = (threadIdx.x < 16 ? P.k_new : P.v_new) + (size_t(b) * P.Hkv + kvh) * kD;
        __nv_bfloat16* dst = (threadIdx.x < 16 ? P.k_pool : P.v_pool) + row * kD;
        reinterpret_cast<uint4*>(dst)[t] = reinterpret_cast<const uint4*>(src)[t];
        fence_proxy_async_global();
      } else if (threadIdx.x == 0) {
        report(P.status, KVSEL_ERR_BAD_INDEX);
      }
      if (threadIdx.x == 0 && P.pos_map)
        P.pos_map[(size_t(b) * P.Hkv + kvh) * P.max_len + S_old] = P.next_pos ? P.next_pos[b] : S_old;
    }
  }
  __syncthreads();

  // per-warp softmax state, used by the consumers (declared here for the merge)
  float m_run = -INFINITY, l_run = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int g = lane >> 2, qd = lane & 3;
  const bool head_ok = g < P.G;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(smem_u32(&empty[s]), ((i / kStages) + 1) & 1, P.status)) break;
        int phys = P.block_table[size_t(b) * P.max_pages + pb + i];
        if (unsigned(phys) >= unsigned(P.num_pages)) {
          report(P.status, KVSEL_ERR_BAD_INDEX);
          phys = 0;
        }
        const int y = (phys * P.Hkv + kvh) * kPage;
        const uint32_t dst = smem_u32(smem + s * kStageBytes);
        const uint32_t bar = smem_u32(&full[s]);
        mbar_expect_tx(bar, kStageBytes);
        tma_load_2d(dst, &tmK, 0, y, bar, pol);
        tma_load_2d(dst + 2048, &tmK, 64, y, bar, pol);
        tma_load_2d(dst + 4096, &tmV, 0, y, bar, pol);
        tma_load_2d(dst + 6144, &tmV, 64, y, bar, pol);
      }
    }
  } else {
    // ---------------- consumers ----------------
    // A fragments of Q (rows = the group's heads, rows 8..15 zero).
    uint32_t qa[8][2];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          P.q + (size_t(b) * P.Hq + kvh * P.G + (head_ok ? g : 0)) * kD);
#pragma unroll
      for (int kt = 0; kt < 8; ++kt) {
        qa[kt][0] = head_ok ? qrow[(16 * kt + 2 * qd) >> 1] : 0u;
        qa[kt][1] = head_ok ? qrow[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
      }
    }
    float* lrow = (P.logits && head_ok)
                      ? P.logits + (size_t(b) * P.Hq + kvh * P.G + g) * P.max_len
                      : nullptr;
    const int mi = lane >> 3, r8 = lane & 7;

#pragma unroll 1
    for (int i = warp; i < n; i += kConsumerWarps) {
      const int s = i % kStages;
      if (!mbar_wait(smem_u32(&full[s]), (i / kStages) & 1, P.status)) break;
      const uint32_t kb = smem_u32(smem + s * kStageBytes);
      const uint32_t vb = kb + 4096;

      // S = Q K^T for 16 keys: n-tile 0 = keys 0..7, n-tile 1 = keys 8..15.
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kt = 0; kt < 8; ++kt) {
        const int key = (mi >> 1) * 8 + r8;
        const int u = 2 * kt + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + tile_off(key, u), b0, b1, b2, b3);
        mma_bf16_16816(s0, qa[kt][0], 0u, qa[kt][1], 0u, b0, b1);
        mma_bf16_16816(s1, qa[kt][0], 0u, qa[kt][1], 0u, b2, b3);
      }
      const int key0 = (pb + i) * kPage;
      const int valid = S - key0;  // >= 1
      const int k0 = 2 * qd, k2 = 8 + 2 * qd;
      const float x0 = k0 < valid ? s0[0] * P.scale_log2 : -INFINITY;
      const float x1 = k0 + 1 < valid ? s0[1] * P.scale_log2 : -INFINITY;
      const float x2 = k2 < valid ? s1[0] * P.scale_log2 : -INFINITY;
      const float x3 = k2 + 1 < valid ? s1[1] * P.scale_log2 : -INFINITY;
      if (lrow) {
        float* dst = lrow + key0;
        if (k0 < valid) dst[k0] = x0;
        if (k0 + 1 < valid) dst[k0 + 1] = x1;
        if (k2 < valid) dst[k2] = x2;
        if (k2 + 1 < valid) dst[k2 + 1] = x3;
      }

      // online softmax (each quad of lanes shares one head row)
      float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = exp2f(m_run - m_new);
      const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
      const float p2 = exp2f(x2 - m_new), p3 = exp2f(x3 - m_new);
      l_run = l_run * alpha + ((p0 + p1) + (p2 + p3));
      m_run = m_new;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= alpha;
        o[nt][1] *= alpha;
        o[nt][2] *= alpha;
        o[nt][3] *= alpha;
      }
      // P as the A operand: rows 0..7 = bf16(p), rows 8..15 = bf16(p - bf16(p)).
      const uint32_t hi01 = pack_bf16x2(p0, p1);
      const uint32_t hi23 = pack_bf16x2(p2, p3);
      const uint32_t lo01 = pack_bf16x2(p0 - bf16lo_to_f32(hi01), p1 - bf16hi_to_f32(hi01));
      const uint32_t lo23 = pack_bf16x2(p2 - bf16lo_to_f32(hi23), p3 - bf16hi_to_f32(hi23));

#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int key = (mi & 1) * 8 + r8;
        const int u = 2 * j + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + tile_off(key, u), b0, b1, b2, b3);
        if (valid < kPage) {  // rows past the live length may hold anything
          b0 = keep_keys(b0, 2 * qd, valid);
          b1 = keep_keys(b1, 8 + 2 * qd, valid);
          b2 = keep_keys(b2, 2 * qd, valid);
          b3 = keep_keys(b3, 8 + 2 * qd, valid);
        }
        mma_bf16_16816(o[2 * j], hi01, lo01, hi23, lo23, b0, b1);
        mma_bf16_16816(o[2 * j + 1], hi01, lo01, hi23, lo23, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  }
  __syncthreads();  // every stage consumed: the ring is free for the merge

  // ---------------- merge the 4 consumer warps ----------------
  float* wo = reinterpret_cast<float*>(smem);                    // [4][8][128]
  float* wm = wo + kConsumerWarps * kMaxG * kD;                  // [4][8]
  float* wl = wm + kConsumerWarps * kMaxG;                       // [4][8]
  if (warp < kConsumerWarps && head_ok) {
    if (qd == 0) {
      wm[warp * kMaxG + g] = m_run;
      wl[warp * kMaxG + g] = l_run;
    }
    float* dst = wo + (warp * kMaxG + g) * kD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      dst[8 * nt + 2 * qd] = o[nt][0] + o[nt][2];
      dst[8 * nt + 2 * qd + 1] = o[nt][1] + o[nt][3];
    }
  }
  __syncthreads();
  const size_t pidx = (size_t(b) * P.Hkv + kvh) * P.splits + split;
  for (int idx = threadIdx.x; idx < P.G * kD; idx += kThreads) {
    const int gg = idx / kD, dd = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wm[w * kMaxG + gg]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = exp2f(wm[w * kMaxG + gg] - M);
        L += wl[w * kMaxG + gg] * f;
        acc += wo[(w * kMaxG + gg) * kD + dd] * f;
      }
    }
    P.part_o[(pidx * P.G + gg) * kD + dd] = acc;
    if (dd == 0) {
      P.part_ml[(pidx * P.G + gg) * 2 + 0] = M;
      P.part_ml[(pidx * P.G + gg) * 2 + 1] = L;
    }
  }
}

struct FinalizeParams {
  const float* part_ml;
  const float* part_o;
  const int32_t* ws_len;
  float* logits;  // in: log2-domain logits; may alias probs
  float* probs;   // out or null
  float* cum;     // in/out or null
  void* out;
  int32_t* seq_lens;
  int32_t* next_pos;
  int out_f32, appended, Hq, Hkv, G, max_len, splits;
};

__global__ void __launch_bounds__(256) decode_finalize_kernel(const FinalizeParams F) {
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int S = F.ws_len[b];
  if (S < 0 || S > F.max_len) return;  // reported by the partial kernel
  __shared__ float sM[kMaxG], sInvL[kMaxG];
  const size_t pbase = (size_t(b) * F.Hkv + kvh) * F.splits;
  if (threadIdx.x < F.G) {
    const int gg = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < F.splits; ++s) M = fmaxf(M, F.part_ml[((pbase + s) * F.G + gg) * 2]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < F.splits; ++s) {
        const float* ml = F.part_ml + ((pbase + s) * F.G + gg) * 2;
        L += ml[1] * exp2f(ml[0] - M);
      }
    sM[gg] = M;
    sInvL[gg] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();

  if (chunk == 0) {
    for (int idx = threadIdx.x; idx < F.G * kD; idx += blockDim.x) {
      const int gg = idx / kD, dd = idx % kD;
      const float M = sM[gg];
      float acc = 0.f;
      if (M != -INFINITY)
        for (int s = 0; s < F.splits; ++s) {
          const float m = F.part_ml[((pbase + s) * F.G + gg) * 2];
          if (m != -INFINITY) acc += F.part_o[((pbase + s) * F.G + gg) * kD + dd] * exp2f(m - M);
        }
      const float v = acc * sInvL[gg];
      const size_t oi = (size_t(b) * F.Hq + kvh * F.G + gg) * kD + dd;
      if (F.out_f32)
        static_cast<float*>(F.out)[oi] = v;
      else
        static_cast<__nv_bfloat16*>(F.out)[oi] = __float2bfloat16_rn(v);
    }
    if (kvh == 0 && threadIdx.x == 0) {
      F.seq_lens[b] = S;
      if (F.appended && F.next_pos) F.next_pos[b] += 1;
    }
  }

  if (!F.logits) return;
  const int j0 = chunk * kFinalizeChunk;
  const int j1 = min(S, j0 + kFinalizeChunk);
  const size_t row0 = (size_t(b) * F.Hq + kvh * F.G) * F.max_len;
  float* crow = F.cum ? F.cum + (size_t(b) * F.Hkv + kvh) * F.max_len : nullptr;
  for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    float sum = 0.f;
    for (int gg = 0; gg < F.G; ++gg) {
      const size_t li = row0 + size_t(gg) * F.max_len + j;
      const float pj = exp2f(F.logits[li] - sM[gg]) * sInvL[gg];
      if (F.probs) F.probs[li] = pj;
      sum += pj;
    }
    if (crow) {
      const float old = (F.appended && j == S - 1) ? 0.f : crow[j];
      crow[j] = old + sum;
    }
  }
}

}  // namespace kvsel

// ---------------------------------------------------------------------------
// host entry points
// ---------------------------------------------------------------------------
using namespace kvsel;
using namespace kvsel_host;

namespace {

struct DecodeWs {
  size_t len_off, ml_off, o_off, logit_off, total;
};

DecodeWs decode_ws_layout(int batch, int Hkv, int Hq, int G, int max_len, bool with_probs) {
  DecodeWs w;
  size_t off = kStatusBytes;
  w.len_off = off;
  off = align_up(off + size_t(batch) * sizeof(int32_t), 256);
  w.ml_off = off;
  off = align_up(off + size_t(batch) * Hkv * kMaxSplits * G * 2 * sizeof(float), 256);
  w.o_off = off;
  off = align_up(off + size_t(batch) * Hkv * kMaxSplits * G * kD * sizeof(float), 256);
  w.logit_off = off;
  if (!with_probs) off = align_up(off + size_t(batch) * Hq * max_len * sizeof(float), 256);
  w.total = off;
  return w;
}

int partial_ctas_per_sm() {
  static int cached = 0;
  if (cached) return cached;
  if (cudaFuncSetAttribute(decode_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kPartialSmem)) != cudaSuccess)
    return 1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_partial_kernel, kThreads,
                                                    kPartialSmem) != cudaSuccess ||
      occ < 1)
    occ = 1;
  cached = occ;
  return occ;
}

}  // namespace

extern "C" size_t kvsel_decode_attn_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                              int with_probs) {
  if (!kv || batch < 1 || max_len < 1 || kv->num_kv_heads < 1 ||
      kv->num_q_heads % kv->num_kv_heads != 0)
    return 0;
  const int G = kv->num_q_heads / kv->num_kv_heads;
  return decode_ws_layout(batch, kv->num_kv_heads, kv->num_q_heads, G, max_len, with_probs != 0).total;
}

extern "C" kvsel_status kvsel_decode_attn(const kvsel_paged_kv* kv, const int32_t* block_table,
                                          int max_pages, int32_t* seq_lens, int batch, const void* q,
                                          const void* k_new, const void* v_new, int32_t* pos_map,
                                          int32_t* next_pos, float scale, void* out, int out_dtype,
                                          float* probs, float* h2o_cum, int max_len, int num_splits,
                                          void* workspace, size_t ws_bytes, void* stream) {
  const char* fn = "kvsel_decode_attn: ";
  if (!kv || !kv->k_pool || !kv->v_pool)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "kv pools must be non-NULL");
  if (kv->head_dim != kD || kv->page_size != kPage)
    return fail(KVSEL_ERR_UNSUPPORTED, std::string(fn) + "only head_dim 128 and page_size 16 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (G > kMaxG)
    return fail(KVSEL_ERR_UNSUPPORTED, std::string(fn) + "at most 8 q heads per kv head are implemented");
  if (kv->num_pages < 1 || (long long)kv->num_pages * Hkv * kPage >= (1LL << 31))
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "num_pages * num_kv_heads * 16 must be in [1, 2^31)");
  if (!block_table || !seq_lens || !q || !out || batch < 1 || max_pages < 1 || max_len < 1)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "block_table, seq_lens, q, out are required; batch, max_pages, max_len >= 1");
  if ((k_new == nullptr) != (v_new == nullptr))
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "k_new and v_new must both be given or both be NULL");
  if (pos_map && !next_pos)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "pos_map needs next_pos");
  if (out_dtype != KVSEL_BF16 && out_dtype != KVSEL_F32)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "out_dtype must be KVSEL_BF16 or KVSEL_F32");
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "num_splits must be in [0, 64]");
  if (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16) || !aligned(q, 16) ||
      (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))))
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "pools, q, k_new, v_new must be 16-byte aligned");
  if (!workspace)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "workspace is required");
  const DecodeWs L = decode_ws_layout(batch, Hkv, Hq, G, max_len, probs != nullptr);
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "workspace too small: need " + std::to_string(L.total));
  if (!aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, std::string(fn) + "workspace must be 256-byte aligned");

  const int pages_max = std::min(max_pages, (max_len + kPage - 1) / kPage);
  int splits = num_splits;
  if (splits == 0) {
    const int slots = sm_count() * partial_ctas_per_sm();
    splits = std::max(1, slots / (batch * Hkv));
    splits = std::min(splits, std::max(1, (pages_max + 7) / 8));
    splits = std::min(splits, kMaxSplits);
  }
  (void)partial_ctas_per_sm();

  CUtensorMap tmK, tmV;
  const uint64_t rows = uint64_t(kv->num_pages) * Hkv * kPage;
  if (!encode_bf16_2d(&tmK, kv->k_pool, kD, rows, kD * 2, 64, kPage) ||
      !encode_bf16_2d(&tmV, kv->v_pool, kD, rows, kD * 2, 64, kPage))
    return fail(KVSEL_ERR_CUDA, std::string(fn) + "tensor-map encode failed");

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* logits = probs ? probs : (h2o_cum ? reinterpret_cast<float*>(ws + L.logit_off) : nullptr);

  DecodeParams P;
  P.block_table = block_table;
  P.seq_lens = seq_lens;
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.k_new = static_cast<const __nv_bfloat16*>(k_new);
  P.v_new = static_cast<const __nv_bfloat16*>(v_new);
  P.k_pool = static_cast<__nv_bfloat16*>(kv->k_pool);
  P.v_pool = static_cast<__nv_bfloat16*>(kv->v_pool);
  P.pos_map = pos_map;
  P.next_pos = next_pos;
  P.logits = logits;
  P.part_ml = reinterpret_cast<float*>(ws + L.ml_off);
  P.part_o = reinterpret_cast<float*>(ws + L.o_off);
  P.ws_len = reinterpret_cast<int32_t*>(ws + L.len_off);
  P.status = reinterpret_cast<int*>(ws);
  P.max_pages = max_pages;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.num_pages = kv->num_pages;
  P.max_len = max_len;
  P.splits = splits;
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  trace_before("decode_partial", st);
  decode_partial_kernel<<<dim3(splits, Hkv, batch), kThreads, kPartialSmem, st>>>(tmK, tmV, P);
  cudaError_t e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_decode_attn (partial launch)");

  FinalizeParams F;
  F.part_ml = P.part_ml;
  F.part_o = P.part_o;
  F.ws_len = P.ws_len;
  F.logits = logits;
  F.probs = probs;
  F.cum = h2o_cum;
  F.out = out;
  F.seq_lens = seq_lens;
  F.next_pos = next_pos;
  F.out_f32 = out_dtype == KVSEL_F32;
  F.appended = k_new != nullptr;
  F.Hq = Hq;
  F.Hkv = Hkv;
  F.G = G;
  F.max_len = max_len;
  F.splits = splits;
  const int chunks = logits ? (max_len + kFinalizeChunk - 1) / kFinalizeChunk : 1;
  trace_before("decode_finalize", st);
  decode_finalize_kernel<<<dim3(chunks, Hkv, batch), 256, 0, st>>>(F);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_decode_attn (finalize launch)");
  return KVSEL_OK;
}
