// DSA-style sparse decode: indexer scores, top-k selection, attention over the
// selected keys only (sm_103a).
//
// What it computes ("Long context, KV eviction and sparse attention": the DSA
// paragraph -- a light few-head indexer scores every past token and each
// query attends only to its best-scored 2048 -- and the sparse-selection
// section's masked softmax):
//   I[b, s] = sum_j w[b, j] * ReLU(q^I[b, j] . k^I[b, s])     for s < S_b
//   sel_b   = the top_k positions by I (ties to the lower position; every
//             position when S_b <= top_k), ascending
//   o[b, h] = softmax over s in sel_b of scale * q[b, h] . K_{h/G}[s], times V
// One selected set per (sequence, step), shared by every q head.
//
// Kernels (four launches on the caller's stream):
//   sd_index_kernel      128 tokens per CTA; the indexer dot products run on
//                        mma.sync (16 tokens x 16 dims x 8 heads per MMA, the
//                        dims permuted per lane so every lane reads 8-byte runs
//                        of a key row); also writes the appended token's K, V
//                        and indexer key.
//   sd_topk_chunk_kernel exact top-k (row_topk) of every 16K-position chunk
//                        of a row, many CTAs per row: the candidates (key and
//                        position, in position order)
//   sd_topk_final_kernel exact top-k of each row over its chunk candidates;
//                        kept positions come out ascending.  (With top_k >=
//                        16K a single sd_topk_kernel per row replaces both.)
//   sd_attn_kernel       (splits, kv head, sequence): each warp gathers 16
//                        selected rows of K and V with cp.async into the
//                        swizzled tile layout (double-buffered; the pages were
//                        resolved by the top-k stage) and runs the shared
//                        mma.sync tile; the 4 warps merge per CTA; the last
//                        split of a (sequence, kv head) merges the splits
//                        into O and the last kv head publishes the length
#include "attn_tile.cuh"
#include "row_topk.cuh"

namespace kvsel {

constexpr int kSdD = 128;
constexpr int kSdPage = 16;
constexpr int kSdDi = 64;
constexpr int kSdMaxHi = 8;
constexpr int kSdTopkGroups = 8;         // rows up to 32K stay in registers; longer rows are swept
constexpr int kSdChunk = 16384;          // positions per first-stage top-k chunk (top_k < kSdChunk)
constexpr int kSdMaxLen = 1 << 28;
constexpr int kSdMaxSplits = kTileMaxSplits;
constexpr int kSdMaxG = kTileMaxG;
constexpr int kSdPartFloats = kPartFloats;
constexpr int kSdAttnWarps = 4;
constexpr size_t kSdAttnSmem = size_t(kSdAttnWarps) * 2 * 8192 + 1024 +
                               size_t(kSdAttnWarps) * kSdMaxG * (kSdD + 2) * 4;

struct SdParams {
  const int32_t* block_table;
  int32_t* seq_lens;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  const __nv_bfloat16* idx_q;      // [B][Hi][64]
  const float* idx_w;              // [B][Hi]
  __nv_bfloat16* idx_k;            // [B][max_len][64]
  const __nv_bfloat16* idx_k_new;  // [B][64] or null
  float* scores;                   // [B][max_len] (workspace or the caller's buffer)
  uint32_t* cand_key;              // [B][nchunks][top_k]: first-stage candidates (two-stage only)
  int32_t* cand_pos;               // [B][nchunks][top_k]
  int32_t* sel;                    // [B][top_k]
  int32_t* sel_page;               // [B][top_k]: physical page of each selected position
  unsigned* merge_cnt;             // [B][Hkv]: splits done (the last one merges)
  unsigned* seq_cnt;               // [B]: kv heads merged (the last one publishes the length)
  int32_t* nsel;                   // [B]
  int32_t* topk_out;               // [B][top_k] or null
  float* part;                     // [B][Hkv][splits][kSdPartFloats]
  void* out;
  int* status;
  int B, max_pages, Hq, Hkv, G, Hi, num_pages, max_len, top_k, nchunks, splits, appended, out_f32;
  float scale_log2;
};

__device__ __forceinline__ bool sd_len_ok(const SdParams& P, int b, int& S) {
  S = P.seq_lens[b] + P.appended;
  return S >= 0 && S <= P.max_len && (S + kSdPage - 1) / kSdPage <= P.max_pages;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) sd_index_kernel(const SdParams P) {
  const int b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int S;
  if (!sd_len_ok(P, b, S)) {
    if (blockIdx.x == 0 && tid == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  const int S_old = S - P.appended;
  if (P.appended && blockIdx.x == 0) {
    // the new token's K, V (every kv head) and indexer key
    const int phys = P.block_table[size_t(b) * P.max_pages + S_old / kSdPage];
    if (unsigned(phys) < unsigned(P.num_pages)) {
      for (int i = tid; i < P.Hkv * 32; i += blockDim.x) {
        const int kvh = i >> 5, t = i & 15;
        const bool isv = (i & 31) >= 16;
        const size_t row = (size_t(phys) * P.Hkv + kvh) * kSdPage + (S_old % kSdPage);
        const uint4* src = reinterpret_cast<const uint4*>((isv ? P.v_new : P.k_new) +
                                                          (size_t(b) * P.Hkv + kvh) * kSdD);
        reinterpret_cast<uint4*>((isv ? P.v_pool : P.k_pool) + row * kSdD)[t] = src[t];
      }
    } else if (tid == 0) {
      report(P.status, KVSEL_ERR_BAD_INDEX);
    }
    if (tid < 8)
      reinterpret_cast<uint4*>(P.idx_k + (size_t(b) * P.max_len + S_old) * kSdDi)[tid] =
          reinterpret_cast<const uint4*>(P.idx_k_new + size_t(b) * kSdDi)[tid];
  }
  const int g = lane >> 2, qd = lane & 3;
  // B fragments: indexer head g (zero past Hi), dims permuted per k-step t:
  // logical k {2q, 2q+1, 2q+8, 2q+9} <-> physical dims 16t + 4q + {0, 1, 2, 3}
  uint32_t bq[4][2];
  const bool h_ok = g < P.Hi;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint2 v = make_uint2(0u, 0u);
    if (h_ok) v = *reinterpret_cast<const uint2*>(P.idx_q + (size_t(b) * P.Hi + g) * kSdDi + 16 * t + 4 * qd);
    bq[t][0] = v.x;
    bq[t][1] = v.y;
  }
  const float w0 = 2 * qd < P.Hi ? P.idx_w[b * P.Hi + 2 * qd] : 0.f;
  const float w1 = 2 * qd + 1 < P.Hi ? P.idx_w[b * P.Hi + 2 * qd + 1] : 0.f;
  float* srow = P.scores + size_t(b) * P.max_len;
#pragma unroll
  for (int grp = 0; grp < 2; ++grp) {
    const int tok0 = blockIdx.x * 128 + warp * 32 + grp * 16;
    if (tok0 >= S) break;
    const int ta = tok0 + g, tb = tok0 + g + 8;
    auto krow = [&](int s) -> const __nv_bfloat16* {
      return (P.appended && s == S_old) ? P.idx_k_new + size_t(b) * kSdDi
                                        : P.idx_k + (size_t(b) * P.max_len + s) * kSdDi;
    };
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint2 va = make_uint2(0u, 0u), vb = make_uint2(0u, 0u);
      if (ta < S) va = *reinterpret_cast<const uint2*>(krow(ta) + 16 * t + 4 * qd);
      if (tb < S) vb = *reinterpret_cast<const uint2*>(krow(tb) + 16 * t + 4 * qd);
      mma_bf16_16816(c, va.x, vb.x, va.y, vb.y, bq[t][0], bq[t][1]);
    }
    float ia = w0 * fmaxf(c[0], 0.f) + w1 * fmaxf(c[1], 0.f);
    float ib = w0 * fmaxf(c[2], 0.f) + w1 * fmaxf(c[3], 0.f);
    ia += __shfl_xor_sync(0xffffffffu, ia, 1);
    ia += __shfl_xor_sync(0xffffffffu, ia, 2);
    ib += __shfl_xor_sync(0xffffffffu, ib, 1);
    ib += __shfl_xor_sync(0xffffffffu, ib, 2);
    if (qd == 0) {
      if (ta < S) srow[ta] = ia;
      if (tb < S) srow[tb] = ib;
    }
  }
}

// ---------------------------------------------------------------------------
// First stage (top_k < kSdChunk): the top_k of every chunk of kSdChunk
// positions (the whole chunk when it is shorter), keys and positions in
// position order.  Every chunk but a row's last holds exactly top_k
// candidates, so a row's candidates are contiguous.
__global__ void __launch_bounds__(kRkThreads) sd_topk_chunk_kernel(const SdParams P) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  RowTopkSmem& sm = *reinterpret_cast<RowTopkSmem*>(tk_smem);
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  int S;
  if (!sd_len_ok(P, b, S)) return;
  const int p0 = c * kSdChunk;
  const int n = max(0, min(kSdChunk, S - p0));
  if (n == 0 || S <= P.top_k) return;
  const int kc = min(P.top_k, n);
  const float* srow = P.scores + size_t(b) * P.max_len + p0;
  uint32_t* ckey = P.cand_key + (size_t(b) * P.nchunks + c) * P.top_k;
  int32_t* cpos = P.cand_pos + (size_t(b) * P.nchunks + c) * P.top_k;
  auto put = [&](int i, int rel) {
    ckey[i] = order_key(__ldcg(srow + rel));
    cpos[i] = p0 + rel;
  };
  if (kc == n) {
    for (int i = tid; i < n; i += kRkThreads) put(i, i);
    return;
  }
  const F32RowKeys src{srow, 0, n, (reinterpret_cast<uintptr_t>(srow) & 15u) == 0};
  row_topk<kSdTopkGroups>(src, kc, 0u, sm, put);
}

// Second stage: the top_k of a row over its chunk candidates, ascending.
__global__ void __launch_bounds__(kRkThreads) sd_topk_final_kernel(const SdParams P) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  RowTopkSmem& sm = *reinterpret_cast<RowTopkSmem*>(tk_smem);
  const int b = blockIdx.x, tid = threadIdx.x;
  int S;
  if (!sd_len_ok(P, b, S)) return;
  const int k = min(P.top_k, S);
  int32_t* sel = P.sel + size_t(b) * P.top_k;
  int32_t* tko = P.topk_out ? P.topk_out + size_t(b) * P.top_k : nullptr;
  int32_t* spage = P.sel_page + size_t(b) * P.top_k;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  auto put = [&](int i, int pos) {
    sel[i] = pos;
    spage[i] = bt[pos / kSdPage];  // resolved once here for every kv head's gather
    if (tko) tko[i] = pos;
  };
  if (k == S) {
    for (int i = tid; i < S; i += kRkThreads) put(i, i);
  } else {
    const int nch = (S + kSdChunk - 1) / kSdChunk;
    const int m = (nch - 1) * P.top_k + min(P.top_k, S - (nch - 1) * kSdChunk);
    const uint32_t* ck = P.cand_key + size_t(b) * P.nchunks * P.top_k;
    const int32_t* cp = P.cand_pos + size_t(b) * P.nchunks * P.top_k;
    const U32RowKeys src{ck, 0, m, (reinterpret_cast<uintptr_t>(ck) & 15u) == 0};
    row_topk<kSdTopkGroups>(src, k, 0u, sm, [&](int i, int rel) { put(i, __ldcg(cp + rel)); });
  }
  if (tko)
    for (int i = k + tid; i < P.top_k; i += kRkThreads) tko[i] = -1;
  if (tid == 0) P.nsel[b] = k;
}

// ---------------------------------------------------------------------------
// Single stage (top_k >= kSdChunk): top-k positions of every row by indexer score (ties to the lower position),
// ascending; every position when S <= top_k.  Also the -1-padded copy for the
// caller.
__global__ void __launch_bounds__(kRkThreads) sd_topk_kernel(const SdParams P) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  RowTopkSmem& sm = *reinterpret_cast<RowTopkSmem*>(tk_smem);
  const int b = blockIdx.x, tid = threadIdx.x;
  int S;
  if (!sd_len_ok(P, b, S)) return;
  const int k = min(P.top_k, S);
  int32_t* sel = P.sel + size_t(b) * P.top_k;
  int32_t* tko = P.topk_out ? P.topk_out + size_t(b) * P.top_k : nullptr;
  int32_t* spage = P.sel_page + size_t(b) * P.top_k;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  auto put = [&](int i, int pos) {
    sel[i] = pos;
    spage[i] = bt[pos / kSdPage];  // resolved once here for every kv head's gather
    if (tko) tko[i] = pos;
  };
  if (k == S) {
    for (int i = tid; i < S; i += kRkThreads) put(i, i);
  } else {
    const float* srow = P.scores + size_t(b) * P.max_len;
    const F32RowKeys src{srow, 0, S, (reinterpret_cast<uintptr_t>(srow) & 15u) == 0};
    row_topk<kSdTopkGroups>(src, k, 0u, sm, put);
  }
  if (tko)
    for (int i = k + tid; i < P.top_k; i += kRkThreads) tko[i] = -1;
  if (tid == 0) P.nsel[b] = k;
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSdAttnWarps * 32) sd_attn_kernel(const SdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* wo = reinterpret_cast<float*>(smem + kSdAttnWarps * 2 * 8192);  // [4][8][130]
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int S;
  if (!sd_len_ok(P, b, S)) return;
  const int nsel = P.nsel[b];
  const int tiles = (nsel + 15) / 16;
  const int t0 = int((long long)split * tiles / P.splits), t1 = int((long long)(split + 1) * tiles / P.splits);
  const int G = P.G, g = lane >> 2, qd = lane & 3;
  const bool head_ok = g < G;
  const int32_t* sel = P.sel + size_t(b) * P.top_k;
  const int32_t* spg = P.sel_page + size_t(b) * P.top_k;
  const uint32_t wbuf = smem_u32(smem + warp * 2 * 8192);

  uint32_t qa[8][2];
  load_q_frags(P.q + (size_t(b) * P.Hq + kvh * G + (head_ok ? g : 0)) * kSdD, head_ok, qd, qa);
  TileState st;
  st.init();

  // gather tile t into stage s: 16 rows of K then 16 of V, 16 x 16-byte units each
  auto gather = [&](int t, int s) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = lane + 32 * i;
      const int row = c >> 4, u = c & 15;  // row 0..31: K rows 0..15, then V rows
      const int r16 = row & 15;
      const int tok = t * 16 + r16;
      const bool valid = tok < nsel;
      const int posi = valid ? sel[tok] : 0;
      int phys = valid ? spg[tok] : 0;
      if (valid && unsigned(phys) >= unsigned(P.num_pages)) {
        report(P.status, KVSEL_ERR_BAD_INDEX);
        phys = 0;
      }
      const __nv_bfloat16* pool = row < 16 ? P.k_pool : P.v_pool;
      const __nv_bfloat16* src =
          pool + ((size_t(phys) * P.Hkv + kvh) * kSdPage + (posi % kSdPage)) * kSdD + u * 8;
      const uint32_t dst = wbuf + s * 8192 + (row < 16 ? 0 : 4096) + tile_unit_off(r16, u);
      cp_async16(dst, src, valid);
    }
    cp_async_commit();
  };

  int t = t0 + warp;
  if (t < t1) gather(t, 0);
  int s = 0;
#pragma unroll 1
  for (; t < t1; t += kSdAttnWarps) {
    const int tn = t + kSdAttnWarps;
    if (tn < t1) {
      gather(tn, s ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    float x0, x1, x2, x3;
    const int valid = min(16, nsel - t * 16);
    attend_tile(wbuf + s * 8192, wbuf + s * 8192 + 4096, qa, valid, P.scale_log2, st, x0, x1, x2, x3);
    __syncwarp();
    s ^= 1;
  }
  float* slot = P.part + ((size_t(b) * P.Hkv + kvh) * P.splits + split) * kSdPartFloats;
  merge_warps_to_slot<kSdAttnWarps>(st, wo, slot, G);
  // The last split of (sequence, kv head) to finish merges all of them into O;
  // the last kv head of a sequence to be merged publishes its length.
  __shared__ int s_last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned done = atomicAdd(P.merge_cnt + size_t(b) * P.Hkv + kvh, 1u) + 1u;
    s_last = done == unsigned(P.splits);
    if (s_last) {
      P.merge_cnt[size_t(b) * P.Hkv + kvh] = 0u;  // every split has arrived: ready for the next call
      __threadfence();
    }
  }
  __syncthreads();
  if (s_last) {
    merge_split_slots(P.part + (size_t(b) * P.Hkv + kvh) * P.splits * kSdPartFloats, P.splits, G, P.out,
                      P.out_f32 != 0, size_t(b) * P.Hq + size_t(kvh) * G, reinterpret_cast<float*>(smem));
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      if (atomicAdd(P.seq_cnt + b, 1u) + 1u == unsigned(P.Hkv)) {
        P.seq_cnt[b] = 0u;
        P.seq_lens[b] = S;  // every CTA of this sequence has read the old length
      }
    }
  }
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct SdWs {
  size_t scores, ckey, cpos, sel, spage, nsel, cnt, part, total;
  int nchunks;  // 0: single-stage top-k
};
SdWs sd_ws_layout(int batch, int Hkv, int max_len, int top_k, bool own_scores) {
  SdWs w;
  w.nchunks = top_k < kSdChunk ? (max_len + kSdChunk - 1) / kSdChunk : 0;
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.scores = own_scores ? take(size_t(batch) * max_len * 4) : 0;
  w.ckey = take(size_t(batch) * w.nchunks * top_k * 4);
  w.cpos = take(size_t(batch) * w.nchunks * top_k * 4);
  w.sel = take(size_t(batch) * top_k * 4);
  w.spage = take(size_t(batch) * top_k * 4);
  w.cnt = take((size_t(batch) * Hkv + batch) * 4);
  w.nsel = take(size_t(batch) * 4);
  w.part = take(size_t(batch) * Hkv * kSdMaxSplits * kSdPartFloats * 4);
  w.total = off;
  return w;
}
}  // namespace

extern "C" size_t kvsel_sparse_decode_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                                int top_k, int with_scores_out) {
  if (!kv || batch < 1 || max_len < 1 || top_k < 1 || kv->num_kv_heads < 1) return 0;
  return sd_ws_layout(batch, kv->num_kv_heads, max_len, top_k, with_scores_out == 0).total;
}

extern "C" kvsel_status kvsel_sparse_decode(const kvsel_paged_kv* kv, const int32_t* block_table,
                                            int max_pages, int32_t* seq_lens, int batch, const void* q,
                                            const void* k_new, const void* v_new, const void* idx_q,
                                            const float* idx_w, void* idx_k, const void* idx_k_new,
                                            int num_idx_heads, int idx_dim, int max_len, int top_k,
                                            float scale, void* out, int out_dtype, int32_t* topk_out,
                                            float* scores_out, void* workspace, size_t ws_bytes,
                                            void* stream) {
  const std::string fn = "kvsel_sparse_decode: ";
  if (!kv || !kv->k_pool || !kv->v_pool)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv pools must be non-NULL");
  if (kv->head_dim != kSdD || kv->page_size != kSdPage)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (G > kSdMaxG) return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 8 q heads per kv head");
  if (idx_dim != kSdDi || num_idx_heads < 1 || num_idx_heads > kSdMaxHi)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "indexer: 1..8 heads of dimension 64 are implemented");
  if (!block_table || !seq_lens || !q || !out || !idx_q || !idx_w || !idx_k || batch < 1 ||
      max_pages < 1 || max_len < 1 || top_k < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "block_table, seq_lens, q, out, idx_q, idx_w, idx_k are "
                                            "required; batch, max_pages, max_len, top_k >= 1");
  if ((k_new == nullptr) != (v_new == nullptr) || (k_new == nullptr) != (idx_k_new == nullptr))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "k_new, v_new and idx_k_new must all be given or all NULL");
  if (out_dtype != KVSEL_BF16 && out_dtype != KVSEL_F32)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "out_dtype must be KVSEL_BF16 or KVSEL_F32");
  const SdWs L = sd_ws_layout(batch, Hkv, max_len, top_k, scores_out == nullptr);
  if (max_len > kSdMaxLen) return fail(KVSEL_ERR_UNSUPPORTED, fn + "max_len must be <= 2^28");
  if (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16) || !aligned(q, 16) || !aligned(idx_k, 16) ||
      !aligned(idx_q, 8) || (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(idx_k_new, 16))))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pools, q, k_new, v_new, idx_k, idx_k_new must be 16-byte aligned");
  if (!workspace || !aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "a 256-byte aligned workspace is required");
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(L.total));

  const int sms = sm_count();
  const int tiles_max = (std::min(top_k, max_len) + 15) / 16;
  int splits = std::max(1, (sms * 4) / (batch * Hkv));
  splits = std::min(splits, std::max(1, (tiles_max + 7) / 8));
  splits = std::min(splits, kSdMaxSplits);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SdParams P;
  P.block_table = block_table;
  P.seq_lens = seq_lens;
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.k_new = static_cast<const __nv_bfloat16*>(k_new);
  P.v_new = static_cast<const __nv_bfloat16*>(v_new);
  P.k_pool = static_cast<__nv_bfloat16*>(kv->k_pool);
  P.v_pool = static_cast<__nv_bfloat16*>(kv->v_pool);
  P.idx_q = static_cast<const __nv_bfloat16*>(idx_q);
  P.idx_w = idx_w;
  P.idx_k = static_cast<__nv_bfloat16*>(idx_k);
  P.idx_k_new = static_cast<const __nv_bfloat16*>(idx_k_new);
  P.scores = scores_out ? scores_out : reinterpret_cast<float*>(ws + L.scores);
  P.cand_key = reinterpret_cast<uint32_t*>(ws + L.ckey);
  P.cand_pos = reinterpret_cast<int32_t*>(ws + L.cpos);
  P.nchunks = L.nchunks;
  P.sel = reinterpret_cast<int32_t*>(ws + L.sel);
  P.sel_page = reinterpret_cast<int32_t*>(ws + L.spage);
  P.merge_cnt = reinterpret_cast<unsigned*>(ws + L.cnt);
  P.seq_cnt = P.merge_cnt + size_t(batch) * Hkv;
  P.nsel = reinterpret_cast<int32_t*>(ws + L.nsel);
  P.topk_out = topk_out;
  P.part = reinterpret_cast<float*>(ws + L.part);
  P.out = out;
  P.status = reinterpret_cast<int*>(ws);
  P.B = batch;
  P.max_pages = max_pages;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.Hi = num_idx_heads;
  P.num_pages = kv->num_pages;
  P.max_len = max_len;
  P.top_k = top_k;
  P.splits = splits;
  P.appended = k_new ? 1 : 0;
  P.out_f32 = out_dtype == KVSEL_F32;
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    cudaError_t e0 = smem_limit_once(reinterpret_cast<const void*>(sd_attn_kernel), int(kSdAttnSmem));
    for (const void* f : {reinterpret_cast<const void*>(sd_topk_kernel),
                          reinterpret_cast<const void*>(sd_topk_chunk_kernel),
                          reinterpret_cast<const void*>(sd_topk_final_kernel)})
      if (e0 == cudaSuccess) e0 = smem_limit_once(f, int(sizeof(RowTopkSmem)));
    if (e0 != cudaSuccess) return cuda_fail(e0, "kvsel_sparse_decode (attribute)");
  }
  cudaError_t e;
#define KVSEL_SD_LAUNCH(name, kernel, grid, block, smem)                 \
  trace_before(name, st);                                                \
  kernel<<<grid, block, smem, st>>>(P);                                  \
  e = cudaGetLastError();                                                \
  trace_after(st);                                                       \
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_sparse_decode (" name ")");
  KVSEL_SD_LAUNCH("sd_index", sd_index_kernel, dim3((max_len + 127) / 128, batch), 128, 0)
  if (L.nchunks > 0) {
    KVSEL_SD_LAUNCH("sd_topk_chunk", sd_topk_chunk_kernel, dim3(L.nchunks, batch), kRkThreads, sizeof(RowTopkSmem))
    KVSEL_SD_LAUNCH("sd_topk_final", sd_topk_final_kernel, dim3(batch), kRkThreads, sizeof(RowTopkSmem))
  } else {
    KVSEL_SD_LAUNCH("sd_topk", sd_topk_kernel, dim3(batch), kRkThreads, sizeof(RowTopkSmem))
  }
  KVSEL_SD_LAUNCH("sd_attn", sd_attn_kernel, dim3(splits, Hkv, batch), kSdAttnWarps * 32, kSdAttnSmem)
#undef KVSEL_SD_LAUNCH
  return KVSEL_OK;
}
