// Score-emitting paged GQA decode attention in one persistent kernel (sm_103a).
//
// What it computes ("From sliding window to attention-guided eviction" §3.1
// and §4.2 step 1; "Long context, KV eviction and sparse attention",
// sparse-selection section): for each sequence and q head, the softmax of the
// scaled logits against every live key, the weighted sum of V, every key's
// probability, and the H2O running score cum[kv head][key] += the sum of the
// group's probabilities.
//
// Layout of the work.  A "unit" is one 16-token page of one (sequence, kv
// head) pair; the units of the whole batch are numbered pair-major and cut
// into gridDim.x equal contiguous ranges, one per CTA (stream-K style: every
// CTA gets the same number of pages whatever the lengths, so a single wave of
// co-resident CTAs finishes together).  A CTA's range covers one or a few
// pairs; each covered piece of a pair is a "segment".
//
// Phase A, per CTA (5 warps):
//   * warp 4 lane 0 is the producer: it walks the range through the block
//     table and TMA-loads each page's K and V rows of its kv head (one 3D
//     load of 4 KB each, two 128-byte-swizzled 64-column halves) into an
//     8-stage ring, evict-first in L2.  The producer's issue loop, not HBM,
//     bounds the stream when a stage takes more instructions, so each stage
//     costs two TMA instructions;
//   * warps 0..3 take pages round-robin: S = Q K^T with mma.sync m16n8k16
//     (A = the group's q rows, at most 8 real; B = 16 keys via ldmatrix),
//     online softmax in the log2 domain, the log2 logits stored to the
//     probability buffer, then O += P V with P split into a bf16 high part
//     (A rows 0..7) and its bf16 residual (rows 8..15), so P keeps ~16
//     mantissa bits at no extra MMA cost;
//   * at each segment end the 4 warps merge and write (m, l, O) for the
//     segment to a partial slot.
// No grid barrier: after phase A a CTA announces each pair it worked on (a
// per-pair counter); phase B of a pair waits (bounded spin; the launch is
// cooperative, so all CTAs are co-resident) only until every owner of that
// pair has announced.
// Phase B, per CTA, for each of its segments: merge the pair's partials into
// (M, L) (every owner's (m, l) fetched at once), write the owner's share of
// O, and turn the segment's stored logits (still in L2) into probabilities
// exp2(s - M) / L, adding the group sum into the H2O score.  The last CTA to
// finish publishes the new lengths.
//
// The CTA that owns the page of a sequence's appended slot writes k_new /
// v_new into the pool (and the slot's original position) before its
// producer starts, fencing the generic-proxy stores against the TMA reads.
#include <mutex>

#include "common.cuh"
#include "h2o_link.cuh"

namespace kvsel {

constexpr int kD = 128;            // head_dim
constexpr int kPage = 16;          // tokens per page
constexpr int kStages = 8;         // TMA ring depth (pages)
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = 8192;  // K (2 x 2 KB swizzled halves) + V (same)
constexpr int kMaxG = 8;
constexpr int kMaxCtas = 1024;
// Consumer warp w takes pages i with i % kConsumerWarps == w, so with a ring
// depth that is a multiple of the warp count a stage is always used by the
// same warp and its parity wait cannot pass on a later lap's phase.
static_assert(kStages % kConsumerWarps == 0, "ring depth must be a multiple of the consumer warps");
constexpr int kMaxBatch = 1024;
constexpr int kPartFloats = kMaxG * (kD + 2);  // one partial slot: m[8], l[8], O[8][128]
constexpr int kMaxOwners = kMaxCtas;           // CTAs sharing one (sequence, kv head) pair

struct SmemLayout {
  static constexpr size_t ring = 0;
  static constexpr size_t merge_o = ring + size_t(kStages) * kStageBytes;                // [4][8][128] f32
  static constexpr size_t merge_ml = merge_o + size_t(kConsumerWarps) * kMaxG * kD * 4;  // [4][8][2] f32
  static constexpr size_t bars = merge_ml + size_t(kConsumerWarps) * kMaxG * 2 * 4;     // 2 x kStages u64
  static constexpr size_t seqS = bars + 2 * kStages * 8;                                 // [kMaxBatch] i32
  static constexpr size_t seqPref = seqS + size_t(kMaxBatch) * 4;                        // [kMaxBatch+1] i64
  static constexpr size_t stats = seqPref + size_t(kMaxBatch + 1) * 8;                   // [8][2] f32
  static constexpr size_t owners = stats + kMaxG * 2 * 4;                                // [kMaxOwners+1] i32
  static constexpr size_t link = owners + (kMaxOwners + 1) * 4;                          // count, base u32
  static constexpr size_t total = link + 2 * 4;
};
// Phase B stages a segment's H2O candidates in the (then idle) TMA ring.
constexpr int kStageCands = kStages * kStageBytes / 8;  // (key u32, slot i32) pairs
// ... and, before that, every owner's partial (m, l) per head.
static_assert(size_t(2) * kMaxOwners * kMaxG * 4 <= size_t(kStages) * kStageBytes, "owner stats fit in the ring");
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack

struct StepParams {
  const int32_t* block_table;
  int32_t* seq_lens;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  int32_t* pos_map;
  int32_t* next_pos;
  float* logits;   // log2-domain logits [B][Hq][max_len] (the probs buffer or workspace), or null
  float* probs;    // output probabilities or null (may alias logits)
  float* cum;      // H2O score [B][Hkv][max_len] or null
  uint32_t* link_hint;   // H2O candidate hand-off (h2o_link.cuh), all null when not linked
  uint32_t* link_count;
  uint32_t* link_key;
  int32_t* link_pos;
  void* out;
  float* part;     // [slots][kPartFloats]
  unsigned* fin;   // CTAs finished (status area); the last one publishes the lengths
  unsigned* pair_cnt;   // [B*Hkv] owners whose phase A is done
  unsigned* pair_pass;  // [B*Hkv] owners past the wait (the last resets both)
  int* status;
  int B, max_pages, Hq, Hkv, G, num_pages, max_len, out_f32;
  int vec_logits;  // logit rows are 8-byte aligned: store pairs as float2
  int vec4;        // logit / score rows are 16-byte aligned: phase B moves float4
  float scale_log2;
};

__device__ __forceinline__ uint32_t tile_off(int key, int u) {
  return (u >> 3) * 2048 + key * 128 + ((((u & 7) ^ (key & 7))) << 4);
}
__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int k0, int valid) {
  return v & ((k0 < valid ? 0x0000FFFFu : 0u) | (k0 + 1 < valid ? 0xFFFF0000u : 0u));
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Bounded spin of one thread until *word == target.  On expiry it records
// KVSEL_ERR_TIMEOUT and returns false (results are then unspecified, but
// nothing hangs).
__device__ __forceinline__ bool wait_word(const unsigned* word, unsigned target, int* status) {
  unsigned spins = 0;
  while (*reinterpret_cast<const volatile unsigned*>(word) != target) {
    __nanosleep(64);
    if (++spins > (1u << 25)) {  // a few seconds
      report(status, KVSEL_ERR_TIMEOUT);
      return false;
    }
  }
  __threadfence();
  return true;
}

struct Locator {
  const int32_t* S;       // live length per sequence (after the append)
  const long long* pref;  // units before sequence b: Hkv * sum_{b'<b} pages(b')
  int B, Hkv;
  __device__ __forceinline__ int pages(int b) const { return (S[b] + kPage - 1) / kPage; }
  // unit u (< total) -> (b, kvh, page)
  __device__ __forceinline__ void locate(long long u, int& b, int& kvh, int& pg) const {
    int lo = 0, hi = B - 1;
    while (lo < hi) {  // last b with pref[b] <= u
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] <= u) lo = mid; else hi = mid - 1;
    }
    b = lo;            // pref is non-decreasing and u < pref[B], so pages(b) > 0 here
    const int np = pages(b);
    const long long r = u - pref[b];
    kvh = int(r / np);
    pg = int(r % np);
  }
};

// The CTA whose range [U*c/NC, U*(c+1)/NC) contains unit u.
__device__ __forceinline__ int cta_of(long long u, long long U, int NC) {
  return int(((u + 1) * NC + U - 1) / U) - 1;
}

// Stages the slots j + c (c < n) whose new score key is >= hk in shared
// memory (sk / sp, counter *scnt): one shared atomic per warp (any subset of
// its lanes).  Entries past kStageCands are dropped; the caller sees the
// overflow in the counter.
template <int n>
__device__ __forceinline__ void link_stage(uint32_t* sk, int32_t* sp, uint32_t* scnt, int j, float4 v,
                                           uint32_t hk) {
  const uint32_t key[4] = {order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w)};
  bool hit[n];
#pragma unroll
  for (int c = 0; c < n; ++c) hit[c] = key[c] >= hk;
  const uint32_t act = __activemask();
  const int lane = threadIdx.x & 31;
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  uint32_t tot = 0, pre = 0;
#pragma unroll
  for (int c = 0; c < n; ++c) {
    const uint32_t b = __ballot_sync(act, hit[c]);
    tot += __popc(b);
    pre += __popc(b & lt);
  }
  if (tot == 0) return;
  const int leader = __ffs(act) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(scnt, tot);
  base = __shfl_sync(act, base, leader) + pre;
#pragma unroll
  for (int c = 0; c < n; ++c)
    if (hit[c]) {
      if (base < uint32_t(kStageCands)) {
        sk[base] = key[c];
        sp[base] = j + c;
      }
      ++base;
    }
}

__global__ void __launch_bounds__(kThreads, 2)
decode_step_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const StepParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* wo = reinterpret_cast<float*>(smem + SmemLayout::merge_o);
  float* wml = reinterpret_cast<float*>(smem + SmemLayout::merge_ml);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemLayout::bars);
  uint64_t* empty = full + kStages;
  int32_t* sS = reinterpret_cast<int32_t*>(smem + SmemLayout::seqS);
  long long* sPref = reinterpret_cast<long long*>(smem + SmemLayout::seqPref);
  float* sStat = reinterpret_cast<float*>(smem + SmemLayout::stats);
  int* sOwn = reinterpret_cast<int*>(smem + SmemLayout::owners);  // [kMaxOwners] + count

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = gridDim.x, c = blockIdx.x;
  const bool append = P.k_new != nullptr;
  const int Hkv = P.Hkv, G = P.G;

  // ---- lengths, unit prefix, this CTA's range ----
  for (int b = tid; b < P.B; b += kThreads) sS[b] = P.seq_lens[b] + (append ? 1 : 0);
  __syncthreads();
  if (tid == 0) {
    long long acc = 0;
    int bad = 0;
    for (int b = 0; b < P.B; ++b) {
      sPref[b] = acc;
      const int S = sS[b];
      const int np = (S + kPage - 1) / kPage;
      if (S < (append ? 1 : 0) || S > P.max_len || np > P.max_pages) bad = 1;
      acc += (long long)Hkv * np;
    }
    sPref[P.B] = bad ? -1 : acc;
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_fence_init();
  }
  if (tid == kConsumerWarps * 32) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncthreads();
  const long long U = sPref[P.B];
  if (U < 0) {  // a length outside the buffers: the same for every CTA, so all leave here
    if (c == 0 && tid == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  const Locator loc{sS, sPref, P.B, Hkv};
  const long long u0 = U * c / NC, u1 = U * (c + 1) / NC;

  // ---- append the new tokens whose page falls in this CTA's range ----
  if (append && tid < 32) {
    for (int b = 0; b < P.B; ++b) {
      const int S_old = sS[b] - 1;
      const int np = loc.pages(b);
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        const long long ua = sPref[b] + (long long)kvh * np + S_old / kPage;
        if (ua < u0 || ua >= u1) continue;
        const int phys = P.block_table[size_t(b) * P.max_pages + S_old / kPage];
        if (unsigned(phys) < unsigned(P.num_pages)) {
          const size_t row = (size_t(phys) * Hkv + kvh) * kPage + (S_old % kPage);
          const int t = tid & 15;
          const __nv_bfloat16* src = (tid < 16 ? P.k_new : P.v_new) + (size_t(b) * Hkv + kvh) * kD;
          __nv_bfloat16* dst = (tid < 16 ? P.k_pool : P.v_pool) + row * kD;
          reinterpret_cast<uint4*>(dst)[t] = reinterpret_cast<const uint4*>(src)[t];
        } else if (tid == 0) {
          report(P.status, KVSEL_ERR_BAD_INDEX);
        }
        if (tid == 0 && P.pos_map)
          P.pos_map[(size_t(b) * Hkv + kvh) * P.max_len + S_old] = P.next_pos ? P.next_pos[b] : S_old;
      }
    }
    fence_proxy_async_global();
  }
  __syncthreads();

  const int n = int(u1 - u0);
  const int g = lane >> 2, qd = lane & 3;
  const bool head_ok = g < G;

  // ================= phase A =================
  if (warp == kConsumerWarps) {
    // Producer warp.  Every lane resolves one page of a 32-page chunk (block
    // table entry -> TMA row coordinate), two chunks ahead of use, so the
    // dependent block-table loads never sit between two TMA issues.
    if (n > 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto resolve = [&](int i) -> int {  // TMA row of CTA-local page i (or -1 past the end)
        if (i >= n) return -1;
        int b, kvh, pg;
        loc.locate(u0 + i, b, kvh, pg);
        int phys = P.block_table[size_t(b) * P.max_pages + pg];
        if (unsigned(phys) >= unsigned(P.num_pages)) {
          report(P.status, KVSEL_ERR_BAD_INDEX);
          phys = 0;
        }
        return (phys * Hkv + kvh) * kPage;
      };
      int y_cur = resolve(lane);
      int y_next = resolve(32 + lane);
#pragma unroll 1
      for (int i0 = 0; i0 < n; i0 += 32) {
        const int y_after = resolve(i0 + 64 + lane);  // issued early; used two chunks later
        bool stop = false;
#pragma unroll 1
        for (int k = 0; k < 32 && i0 + k < n; ++k) {
          const int i = i0 + k;
          const int y = __shfl_sync(0xffffffffu, y_cur, k);
          const int s = i % kStages;
          bool ok = true;
          if (i >= kStages) ok = mbar_wait(smem_u32(&empty[s]), ((i / kStages) + 1) & 1, P.status);
          if (!__all_sync(0xffffffffu, ok)) {
            stop = true;
            break;
          }
          if (lane == 0) {
            const uint32_t dst = smem_u32(smem + SmemLayout::ring + s * kStageBytes);
            const uint32_t bar = smem_u32(&full[s]);
            mbar_expect_tx(bar, kStageBytes);
            tma_load_3d(dst, &tmK, 0, y, 0, bar, pol);
            tma_load_3d(dst + 4096, &tmV, 0, y, 0, bar, pol);
          }
          __syncwarp();
        }
        if (stop) break;
        y_cur = y_next;
        y_next = y_after;
      }
    }
  } else {
    const int mi = lane >> 3, r8 = lane & 7;
    long long u = u0;
#pragma unroll 1
    while (u < u1) {
      int b, kvh, pg;
      loc.locate(u, b, kvh, pg);
      const int S = sS[b];
      const int np = loc.pages(b);
      const long long seg_end = min(u1, u + (np - pg));
      const int pair = b * Hkv + kvh;

      uint32_t qa[8][2];
      {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            P.q + (size_t(b) * P.Hq + kvh * G + (head_ok ? g : 0)) * kD);
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          qa[kt][0] = head_ok ? qrow[(16 * kt + 2 * qd) >> 1] : 0u;
          qa[kt][1] = head_ok ? qrow[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
        }
      }
      float* lrow = (P.logits && head_ok)
                        ? P.logits + (size_t(b) * P.Hq + kvh * G + g) * P.max_len
                        : nullptr;
      float m_run = -INFINITY, l_run = 0.f;
      float o[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

      const int i_begin = int(u - u0), i_end = int(seg_end - u0);
      // first index >= i_begin that belongs to this warp (index % 4 == warp)
      int i = i_begin + ((warp - i_begin) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
#pragma unroll 1
      for (; i < i_end; i += kConsumerWarps) {
        const int s = i % kStages;
        if (!mbar_wait(smem_u32(&full[s]), (i / kStages) & 1, P.status)) break;
        const uint32_t kb = smem_u32(smem + SmemLayout::ring + s * kStageBytes);
        const uint32_t vb = kb + 4096;

        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          const int key = (mi >> 1) * 8 + r8;
          const int uu = 2 * kt + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + tile_off(key, uu), b0, b1, b2, b3);
          mma_bf16_16816(s0, qa[kt][0], 0u, qa[kt][1], 0u, b0, b1);
          mma_bf16_16816(s1, qa[kt][0], 0u, qa[kt][1], 0u, b2, b3);
        }
        const int key0 = (pg + (i - i_begin)) * kPage;
        const int valid = S - key0;  // >= 1
        const int k0 = 2 * qd, k2 = 8 + 2 * qd;
        const float x0 = k0 < valid ? s0[0] * P.scale_log2 : -INFINITY;
        const float x1 = k0 + 1 < valid ? s0[1] * P.scale_log2 : -INFINITY;
        const float x2 = k2 < valid ? s1[0] * P.scale_log2 : -INFINITY;
        const float x3 = k2 + 1 < valid ? s1[1] * P.scale_log2 : -INFINITY;
        if (lrow) {
          float* dst = lrow + key0;
          if (valid >= kPage && P.vec_logits) {
            *reinterpret_cast<float2*>(dst + k0) = make_float2(x0, x1);
            *reinterpret_cast<float2*>(dst + k2) = make_float2(x2, x3);
          } else {
            if (k0 < valid) dst[k0] = x0;
            if (k0 + 1 < valid) dst[k0 + 1] = x1;
            if (k2 < valid) dst[k2] = x2;
            if (k2 + 1 < valid) dst[k2 + 1] = x3;
          }
        }
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
        const uint32_t hi01 = pack_bf16x2(p0, p1);
        const uint32_t hi23 = pack_bf16x2(p2, p3);
        const uint32_t lo01 = pack_bf16x2(p0 - bf16lo_to_f32(hi01), p1 - bf16hi_to_f32(hi01));
        const uint32_t lo23 = pack_bf16x2(p2 - bf16lo_to_f32(hi23), p3 - bf16hi_to_f32(hi23));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int key = (mi & 1) * 8 + r8;
          const int uu = 2 * j + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + tile_off(key, uu), b0, b1, b2, b3);
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

      // ---- merge the 4 warps' state of this segment into partial slot c + pair ----
      if (head_ok) {
        if (qd == 0) {
          wml[(warp * kMaxG + g) * 2 + 0] = m_run;
          wml[(warp * kMaxG + g) * 2 + 1] = l_run;
        }
        float* dst = wo + (warp * kMaxG + g) * kD;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) =
              make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
      }
      consumer_sync();
      float* slot = P.part + size_t(c + pair) * kPartFloats;
      for (int idx = tid; idx < G * kD; idx += kConsumerWarps * 32) {
        const int gg = idx / kD, dd = idx % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wml[(w * kMaxG + gg) * 2]);
        float L = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = exp2f(wml[(w * kMaxG + gg) * 2] - M);
            L += wml[(w * kMaxG + gg) * 2 + 1] * f;
            acc += wo[(w * kMaxG + gg) * kD + dd] * f;
          }
        }
        slot[2 * kMaxG + gg * kD + dd] = acc;
        if (dd == 0) {
          slot[gg] = M;
          slot[kMaxG + gg] = L;
        }
      }
      consumer_sync();
      u = seg_end;
    }
  }

  // ---- announce: this CTA's partials (and logits) for its pairs are written ----
  // No grid barrier: phase B of a pair waits only for that pair's owners.
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (long long u = u0; u < u1;) {
      int b, kvh, pg;
      loc.locate(u, b, kvh, pg);
      const int pair = b * Hkv + kvh;
      // the first owner gives the pair a fresh H2O candidate list before anyone can append
      if (P.link_count && pg == 0) P.link_count[pair] = 0u;
      __threadfence();
      atomicAdd(P.pair_cnt + pair, 1u);
      u = min(u1, u + (loc.pages(b) - pg));
    }
  }

  // ================= phase B =================
  uint32_t* sLink = reinterpret_cast<uint32_t*>(smem + SmemLayout::link);  // staged count, list base
  uint32_t* stKey = reinterpret_cast<uint32_t*>(smem + SmemLayout::ring);  // the idle TMA ring
  int32_t* stPos = reinterpret_cast<int32_t*>(smem + SmemLayout::ring + kStageCands * 4);
  if (c == 0) {
    for (int b = 0; b < P.B; ++b)  // sequences without keys: O = 0
      if (sS[b] == 0)
        for (int idx = tid; idx < P.Hq * kD; idx += kThreads) {
          const size_t oi = size_t(b) * P.Hq * kD + idx;
          if (P.out_f32) static_cast<float*>(P.out)[oi] = 0.f;
          else static_cast<__nv_bfloat16*>(P.out)[oi] = __float2bfloat16_rn(0.f);
        }
  }
  long long u = u0;
#pragma unroll 1
  while (u < u1) {
    int b, kvh, pg;
    loc.locate(u, b, kvh, pg);
    const int S = sS[b];
    const int np = loc.pages(b);
    const long long seg_end = min(u1, u + (np - pg));
    const int pair = b * Hkv + kvh;
    const long long pfirst = sPref[b] + (long long)kvh * np, plast = pfirst + np - 1;
    const int cf = cta_of(pfirst, U, NC);
    // The CTAs owning units of this pair, in order: cf, then the owner of the
    // unit right after each owner's range, up to the pair's last unit.
    if (tid == 0) {
      int no = 0;
      for (int cc = cf; cc >= 0 && no < kMaxOwners; ++no) {
        sOwn[no] = cc;
        const long long nu = U * (cc + 1) / NC;
        cc = nu > plast ? -1 : cta_of(nu, U, NC);
      }
      sOwn[kMaxOwners] = no;
      sLink[0] = 0u;
      // every owner of the pair has announced: its partials are complete
      if (wait_word(P.pair_cnt + pair, unsigned(no), P.status) &&
          atomicAdd(P.pair_pass + pair, 1u) + 1u == unsigned(no)) {
        P.pair_cnt[pair] = 0u;  // every owner is past the wait: reset for the next launch
        P.pair_pass[pair] = 0u;
      }
    }
    __syncthreads();
    const int nown = sOwn[kMaxOwners];
    // every owner's (m, l) per head, fetched in parallel into the idle TMA ring
    float* sM = reinterpret_cast<float*>(smem + SmemLayout::ring);  // [kMaxOwners][kMaxG]
    float* sL = sM + kMaxOwners * kMaxG;
    for (int i = tid; i < nown * G; i += kThreads) {
      const int k = i / G, g = i - k * G;
      const float* sl = P.part + size_t(sOwn[k] + pair) * kPartFloats;
      sM[k * kMaxG + g] = __ldcg(sl + g);
      sL[k * kMaxG + g] = __ldcg(sl + kMaxG + g);
    }
    __syncthreads();
    if (tid < G) {
      float M = -INFINITY;
      for (int k = 0; k < nown; ++k) M = fmaxf(M, sM[k * kMaxG + tid]);
      float L = 0.f;
      for (int k = 0; k < nown; ++k) {
        const float m = sM[k * kMaxG + tid];
        if (m != -INFINITY) L += sL[k * kMaxG + tid] * exp2f(m - M);
      }
      sStat[tid * 2] = M;
      sStat[tid * 2 + 1] = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    {  // O = the rescaled sum of the partials: each owner merges its share of the G x 128 outputs
      int kme = 0;
      while (kme < nown - 1 && sOwn[kme] != c) ++kme;
      const int E = G * kD;
      const int e1 = (kme + 1) * E / nown;
      for (int idx = kme * E / nown + tid; idx < e1; idx += kThreads) {
        const int gg = idx / kD, dd = idx % kD;
        const float M = sStat[gg * 2];
        float acc = 0.f;
#pragma unroll 4
        for (int k = 0; k < nown; ++k) {
          const float m = sM[k * kMaxG + gg];
          if (m != -INFINITY)
            acc += __ldcg(P.part + size_t(sOwn[k] + pair) * kPartFloats + 2 * kMaxG + gg * kD + dd) * exp2f(m - M);
        }
        const float v = acc * sStat[gg * 2 + 1];
        const size_t oi = (size_t(b) * P.Hq + kvh * G + gg) * kD + dd;
        if (P.out_f32) static_cast<float*>(P.out)[oi] = v;
        else static_cast<__nv_bfloat16*>(P.out)[oi] = __float2bfloat16_rn(v);
      }
    }
    __syncthreads();  // the ring is reused for the H2O candidate stage below
    if (P.logits) {
      const int j0 = pg * kPage;
      const int j1 = min(S, int(pg + (seg_end - u)) * kPage);
      const size_t row0 = (size_t(b) * P.Hq + kvh * G) * P.max_len;
      float* crow = P.cum ? P.cum + (size_t(b) * Hkv + kvh) * P.max_len : nullptr;
      // the row's last H2O threshold: collect the slots at or above it (0: no list)
      const uint32_t hk = (crow && P.link_hint) ? __ldcg(P.link_hint + pair) : 0u;
      float Mg[kMaxG], Ig[kMaxG];
#pragma unroll
      for (int gg = 0; gg < kMaxG; ++gg) {
        Mg[gg] = gg < G ? sStat[gg * 2] : 0.f;
        Ig[gg] = gg < G ? sStat[gg * 2 + 1] : 0.f;
      }
      if (P.vec4) {
        // 4 keys x all heads per thread, two such groups per iteration: up to 16
        // independent 16-byte loads in flight per thread (a third group would
        // not fit the 168 registers that two CTAs per SM leave each thread)
        auto group = [&](int j, float4 (&lg)[kMaxG]) {
#pragma unroll
          for (int gg = 0; gg < kMaxG; ++gg)
            if (gg < G)
              lg[gg] = __ldcg(reinterpret_cast<const float4*>(P.logits + row0 + size_t(gg) * P.max_len + j));
        };
        auto finish = [&](int j, const float4 (&lg)[kMaxG], float4 old) {
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int gg = 0; gg < kMaxG; ++gg)
            if (gg < G) {
              float4 pj;
              pj.x = exp2f(lg[gg].x - Mg[gg]) * Ig[gg];
              pj.y = exp2f(lg[gg].y - Mg[gg]) * Ig[gg];
              pj.z = exp2f(lg[gg].z - Mg[gg]) * Ig[gg];
              pj.w = exp2f(lg[gg].w - Mg[gg]) * Ig[gg];
              if (P.probs) __stcg(reinterpret_cast<float4*>(P.probs + row0 + size_t(gg) * P.max_len + j), pj);
              sum.x += pj.x;
              sum.y += pj.y;
              sum.z += pj.z;
              sum.w += pj.w;
            }
          if (crow) {
            if (append && j + 3 >= S - 1) {  // the appended slot starts from zero
              if (j == S - 1) old.x = 0.f;
              if (j + 1 == S - 1) old.y = 0.f;
              if (j + 2 == S - 1) old.z = 0.f;
              if (j + 3 == S - 1) old.w = 0.f;
            }
            const float4 nv = make_float4(old.x + sum.x, old.y + sum.y, old.z + sum.z, old.w + sum.w);
            __stcg(reinterpret_cast<float4*>(crow + j), nv);
            if (hk) link_stage<4>(stKey, stPos, sLink, j, nv, hk);
          }
        };
        const int jend = j0 + ((j1 - j0) & ~3);
        for (int j = j0 + 4 * tid; j < jend; j += 8 * kThreads) {
          const int jb = j + 4 * kThreads;
          const bool has_b = jb < jend;
          float4 la[kMaxG], lb[kMaxG];
          group(j, la);
          if (has_b) group(jb, lb);
          float4 oa = make_float4(0.f, 0.f, 0.f, 0.f), ob = oa;
          if (crow) {
            oa = __ldcg(reinterpret_cast<const float4*>(crow + j));
            if (has_b) ob = __ldcg(reinterpret_cast<const float4*>(crow + jb));
          }
          finish(j, la, oa);
          if (has_b) finish(jb, lb, ob);
        }
      }
      // keys left over (the whole segment when rows are not 16-byte aligned), one per thread
      const int jr = P.vec4 ? j0 + ((j1 - j0) & ~3) : j0;
      for (int jj = jr + tid; jj < j1; jj += kThreads) {
        float sum = 0.f;
#pragma unroll
        for (int gg = 0; gg < kMaxG; ++gg)
          if (gg < G) {
            const size_t li = row0 + size_t(gg) * P.max_len + jj;
            const float pj = exp2f(__ldcg(P.logits + li) - Mg[gg]) * Ig[gg];
            if (P.probs) P.probs[li] = pj;
            sum += pj;
          }
        if (crow) {
          const float old = (append && jj == S - 1) ? 0.f : crow[jj];
          const float nv = old + sum;
          crow[jj] = nv;
          if (hk) link_stage<1>(stKey, stPos, sLink, jj, make_float4(nv, 0.f, 0.f, 0.f), hk);
        }
      }
      if (hk) {  // hand this segment's candidates to the row's list: one global atomic
        __syncthreads();
        const uint32_t n = sLink[0];
        if (tid == 0)  // an overflowing stage invalidates the row's list (count > capacity)
          sLink[1] = atomicAdd(P.link_count + pair, n > uint32_t(kStageCands) ? uint32_t(kLinkCap) + 1u : n);
        __syncthreads();
        const uint32_t base = sLink[1];
        if (n <= uint32_t(kStageCands)) {
          uint32_t* gk = P.link_key + size_t(pair) * kLinkCap;
          int32_t* gp = P.link_pos + size_t(pair) * kLinkCap;
          for (uint32_t i = tid; i < n && base + i < uint32_t(kLinkCap); i += kThreads) {
            gk[base + i] = stKey[i];
            gp[base + i] = stPos[i];
          }
        }
      }
    }
    __syncthreads();
    u = seg_end;
  }
  // The last CTA to finish publishes the new lengths: every CTA has read the
  // old ones by then.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.fin, 1u) + 1u == unsigned(NC)) {
      *P.fin = 0u;
      for (int b = 0; b < P.B; ++b) {
        P.seq_lens[b] = sS[b];
        if (append && P.next_pos) P.next_pos[b] += 1;
      }
      __threadfence();
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
  size_t pair_off, part_off, logit_off, total;
};

// The finish counter lives in the workspace's status area (byte 64); the
// per-pair readiness counters follow it.
DecodeWs decode_ws_layout(int batch, int Hkv, int Hq, int max_len, bool with_probs) {
  DecodeWs w;
  size_t off = kStatusBytes;
  w.pair_off = off;
  off = align_up(off + size_t(batch) * Hkv * 2 * sizeof(unsigned), 256);
  w.part_off = off;
  off = align_up(off + (size_t(kMaxCtas) + size_t(batch) * Hkv) * kPartFloats * sizeof(float), 256);
  w.logit_off = off;
  if (!with_probs) off = align_up(off + size_t(batch) * Hq * max_len * sizeof(float), 256);
  w.total = off;
  return w;
}

int ctas_per_sm() {
  static int cached = 0;
  if (cached) return cached;
  if (cudaFuncSetAttribute(decode_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemBytes)) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_step_kernel, kThreads, kSmemBytes) !=
      cudaSuccess)
    return 0;
  cached = occ;
  return occ;
}

}  // namespace

extern "C" size_t kvsel_decode_attn_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                              int with_probs) {
  if (!kv || batch < 1 || max_len < 1 || kv->num_kv_heads < 1 ||
      kv->num_q_heads % kv->num_kv_heads != 0)
    return 0;
  return decode_ws_layout(batch, kv->num_kv_heads, kv->num_q_heads, max_len, with_probs != 0).total;
}

extern "C" kvsel_status kvsel_decode_attn(const kvsel_paged_kv* kv, const int32_t* block_table,
                                          int max_pages, int32_t* seq_lens, int batch, const void* q,
                                          const void* k_new, const void* v_new, int32_t* pos_map,
                                          int32_t* next_pos, float scale, void* out, int out_dtype,
                                          float* probs, float* h2o_cum, int max_len, int num_ctas,
                                          void* workspace, size_t ws_bytes, void* h2o_link,
                                          size_t h2o_link_bytes, void* stream) {
  const std::string fn = "kvsel_decode_attn: ";
  if (!kv || !kv->k_pool || !kv->v_pool)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv pools must be non-NULL");
  if (kv->head_dim != kD || kv->page_size != kPage)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (G > kMaxG) return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 8 q heads per kv head are implemented");
  if (kv->num_pages < 1 || (long long)kv->num_pages * Hkv * kPage >= (1LL << 31))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_pages * num_kv_heads * 16 must be in [1, 2^31)");
  if (!block_table || !seq_lens || !q || !out || batch < 1 || max_pages < 1 || max_len < 1)
    return fail(KVSEL_ERR_INVALID_ARG,
                fn + "block_table, seq_lens, q, out are required; batch, max_pages, max_len >= 1");
  if (batch > kMaxBatch)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 1024 sequences per call are implemented");
  if ((k_new == nullptr) != (v_new == nullptr))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "k_new and v_new must both be given or both be NULL");
  if (pos_map && !next_pos) return fail(KVSEL_ERR_INVALID_ARG, fn + "pos_map needs next_pos");
  if (out_dtype != KVSEL_BF16 && out_dtype != KVSEL_F32)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "out_dtype must be KVSEL_BF16 or KVSEL_F32");
  if (num_ctas < 0 || num_ctas > kMaxCtas)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_ctas must be in [0, 1024]");
  if (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16) || !aligned(q, 16) ||
      (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pools, q, k_new, v_new must be 16-byte aligned");
  if (probs && !aligned(probs, 4)) return fail(KVSEL_ERR_INVALID_ARG, fn + "probs must be 4-byte aligned");
  if (!workspace) return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace is required");
  const DecodeWs L = decode_ws_layout(batch, Hkv, Hq, max_len, probs != nullptr);
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(L.total));
  if (!aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace must be 256-byte aligned");
  if (h2o_link && (!aligned(h2o_link, 256) || h2o_link_bytes < link_bytes(batch * Hkv)))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "h2o_link must be a 256-byte aligned H2O evict workspace of at least " +
                                           std::to_string(link_bytes(batch * Hkv)) + " bytes");

  const int occ = ctas_per_sm();
  if (occ < 1) return fail(KVSEL_ERR_CUDA, fn + "cannot configure the decode kernel (occupancy 0)");
  const int resident = sm_count() * occ;
  const int nc = num_ctas == 0 ? std::min(resident, kMaxCtas) : num_ctas;
  if (nc > resident)
    return fail(KVSEL_ERR_INVALID_ARG,
                fn + "num_ctas exceeds the co-resident CTA count " + std::to_string(resident));

  CUtensorMap tmK, tmV;
  const uint64_t rows = uint64_t(kv->num_pages) * Hkv * kPage;
  if (!encode_bf16_row_pages(&tmK, kv->k_pool, rows, kPage) ||
      !encode_bf16_row_pages(&tmV, kv->v_pool, rows, kPage))
    return fail(KVSEL_ERR_CUDA, fn + "tensor-map encode failed");

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  StepParams P;
  P.block_table = block_table;
  P.seq_lens = seq_lens;
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.k_new = static_cast<const __nv_bfloat16*>(k_new);
  P.v_new = static_cast<const __nv_bfloat16*>(v_new);
  P.k_pool = static_cast<__nv_bfloat16*>(kv->k_pool);
  P.v_pool = static_cast<__nv_bfloat16*>(kv->v_pool);
  P.pos_map = pos_map;
  P.next_pos = next_pos;
  P.logits = probs ? probs : (h2o_cum ? reinterpret_cast<float*>(ws + L.logit_off) : nullptr);
  P.probs = probs;
  P.cum = h2o_cum;
  P.link_hint = P.link_count = P.link_key = nullptr;
  P.link_pos = nullptr;
  if (h2o_link && h2o_cum) {
    const H2OLink L2 = link_layout(h2o_link, batch * Hkv);
    P.link_hint = L2.hint;
    P.link_count = L2.count;
    P.link_key = L2.key;
    P.link_pos = L2.pos;
  }
  P.out = out;
  P.part = reinterpret_cast<float*>(ws + L.part_off);
  P.fin = reinterpret_cast<unsigned*>(ws + 64);
  P.pair_cnt = reinterpret_cast<unsigned*>(ws + L.pair_off);
  P.pair_pass = P.pair_cnt + size_t(batch) * Hkv;
  P.status = reinterpret_cast<int*>(ws);
  P.B = batch;
  P.max_pages = max_pages;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.num_pages = kv->num_pages;
  P.max_len = max_len;
  P.out_f32 = out_dtype == KVSEL_F32;
  P.vec_logits = (max_len % 2 == 0) && aligned(P.logits, 8);
  P.vec4 = (max_len % 4 == 0) && aligned(P.logits, 16) && (!h2o_cum || aligned(h2o_cum, 16));
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before("decode_step", st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_step_kernel, tmK, tmV, P);
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_decode_attn (launch)");
  return KVSEL_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of kvsel_decode_attn.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: an allocator-less runtime embedding this library, a plug-in
// whose host owns every allocation, or code that must not touch the
// allocator mid-step.  For them the scratch the decode kernel needs (status
// and readiness counters, per-CTA partial results, and the logit buffer when
// no probability buffer is given) lives in the fixed array below, which every
// GPU that loads this library holds until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
}  // namespace

extern "C" kvsel_status kvsel_decode_attn_noalloc(const kvsel_paged_kv* kv, const int32_t* block_table,
                                                  int max_pages, int32_t* seq_lens, int batch,
                                                  const void* q, const void* k_new, const void* v_new,
                                                  int32_t* pos_map, int32_t* next_pos, float scale,
                                                  void* out, int out_dtype, float* probs, float* h2o_cum,
                                                  int max_len, int num_ctas, void* stream) {
  const std::string fn = "kvsel_decode_attn_noalloc: ";
  if (!kv || batch < 1 || max_len < 1 || kv->num_kv_heads < 1 || kv->num_q_heads < 1 ||
      kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv descriptor, batch >= 1 and max_len >= 1 are required");
  const size_t need = decode_ws_layout(batch, kv->num_kv_heads, kv->num_q_heads, max_len,
                                       probs != nullptr).total;
  if (need > kNoAllocScratchBytes)
    return fail(KVSEL_ERR_INVALID_ARG,
                fn + "this call needs " + std::to_string(need) + " bytes of scratch, more than the " +
                    std::to_string(kNoAllocScratchBytes) +
                    "-byte built-in array (pass a probs buffer, or use kvsel_decode_attn with a workspace)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_decode_attn_noalloc (cudaGetDevice)");
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "device ordinal above 63");
  void* scratch = nullptr;
  {
    // Set-up, once per device, with that device current: the array's name is
    // only a host-side stand-in; the kernel needs its device address.
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e, "kvsel_decode_attn_noalloc (cudaGetSymbolAddress)");
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The status word and the finish / per-pair readiness counters must start at
  // zero; the array keeps whatever the previous call left there.
  const size_t counters = decode_ws_layout(batch, kv->num_kv_heads, kv->num_q_heads, max_len,
                                           probs != nullptr).part_off;
  e = cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_decode_attn_noalloc (clear)");
  return kvsel_decode_attn(kv, block_table, max_pages, seq_lens, batch, q, k_new, v_new, pos_map,
                           next_pos, scale, out, out_dtype, probs, h2o_cum, max_len, num_ctas, scratch,
                           kNoAllocScratchBytes, nullptr, 0, stream);
}
