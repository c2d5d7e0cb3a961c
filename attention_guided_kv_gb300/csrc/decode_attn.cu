// Score-emitting paged GQA decode attention in one persistent kernel (sm_103a).
//
// What it computes ("From sliding window to attention-guided eviction" §3.1
// and §4.2 step 1; "Long context, KV eviction and sparse attention",
// sparse-selection section): for each sequence and q head, the softmax of the
// scaled logits against every live key, the weighted sum of V, every key's
// probability, and the H2O running score cum[kv head][key] += the sum of the
// group's probabilities.
//
// Layout of the work.  A "unit" is one 16-token tile of one (sequence, kv
// head) pair: a whole page of a 16-token pool, or one of the 2..16 tiles of
// a larger page (pools of 32..256-token pages).  The units of the whole
// batch are numbered pair-major and cut into gridDim.x equal contiguous
// ranges, one per CTA (stream-K style: every CTA gets the same number of
// tiles whatever the lengths, so a single wave of co-resident CTAs finishes
// together).  A CTA's range covers one or a few
// pairs; each covered piece of a pair is a "segment".
//
// Each CTA (6 warps) streams its range twice, K pages first, then V pages:
// warps 4 and 5 are producers, TMA-loading two pages of K (or of V) of its
// kv head per 8 KB stage -- one 3D load per 4 KB page, two 128-byte-swizzled
// 64-column halves -- into an 8-stage ring, evict-first in L2, alternating
// stages; warps 0..3 take the ring's stages round-robin.  (A producer's
// issue loop costs a fixed few hundred cycles per stage, so one-page stages
// or a single producer warp could not keep up with HBM.)
//   * K pass: S = Q K^T with mma.sync m16n8k16 (A = the group's q rows, up
//     to 16: head g in row g, head g + 8 in row g + 8; B = 16 keys via
//     ldmatrix); the scaled log2-domain logits
//     are stored to the probability buffer, marked evict-last so they are
//     still in L2 for the V pass, and each lane keeps a running (max, sum of
//     exp2) of its keys.  At a segment end the CTA writes the segment's
//     (m, l) per head to a partial slot and announces the pair (a per-pair
//     counter).
//   * V pass: per segment, once every owner of the pair has announced
//     (bounded spin; the grid is at most the co-resident CTA count, and by
//     the end of a K pass every CTA has started),
//     the pair's exact (M, L) per head are merged from the owners' slots.
//     Every page then turns its stored logits into final probabilities
//     p = exp2(s - M) / L, writes them (evict-first), adds the group's sum
//     into the H2O score (collecting the H2O candidates of the next
//     selection), and
//     accumulates O += P V with P split into a bf16 high part and its bf16
//     residual, so P keeps ~16 mantissa bits: with up to 8 heads the high
//     parts fill A rows 0..7 and the residuals rows 8..15 (no extra MMA);
//     with more, a second MMA adds the residuals.  The segment's O, already normalised, is added into
//     the pair's fp32 accumulator; the owner that adds last writes O and
//     clears the accumulator, so no owner waits for another at the end.
// The normalisation work therefore overlaps the V stream instead of trailing
// the kernel.
//
// The CTA that owns the page of a sequence's appended slot writes k_new /
// v_new into the pool (and the slot's original position) before its
// producer starts, fencing the generic-proxy stores against the TMA reads.
// Once every CTA is past that point, the last one publishes the new lengths.
#include <mutex>

#include "common.cuh"
#include "h2o_link.cuh"

namespace kvsel {

constexpr int kD = 128;            // head_dim
constexpr int kPage = 16;          // tokens per page
constexpr int kStages = 8;         // TMA ring depth (two pages of K or of V per stage)
constexpr int kConsumerWarps = 4;
constexpr int kProducerWarps = 2;  // alternate stages: the issue loop's fixed cost is halved per warp
constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kPageBytes = 4096;   // 16 rows x 128 bf16, as two 2 KB swizzled halves
constexpr int kStageBytes = 2 * kPageBytes;
constexpr int kMaxG = 16;   // q heads per kv head: rows g and g + 8 of the MMA tiles
constexpr int kRowG = 8;    // q heads whose O one merge round moves (the A tile's first 8 rows)
constexpr int kMaxCtas = 1024;
// Consumer warp w takes the stages t with t % kConsumerWarps == w, so with a
// ring depth that is a multiple of the warp count a stage is always used by
// the same warp and its parity wait cannot pass on a later lap's phase.
static_assert(kStages % kConsumerWarps == 0, "ring depth must be a multiple of the consumer warps");
static_assert(kStages % kProducerWarps == 0, "a ring slot must always have the same producer");
constexpr int kMaxBatch = 1024;
constexpr int kPartFloats = 2 * kMaxG;  // one partial slot: m[16], l[16] of an owner's segment
constexpr int kMaxOwners = kMaxCtas;           // CTAs sharing one (sequence, kv head) pair
constexpr int kWarpCands = 256;                // H2O candidates a consumer warp stages

struct SmemLayout {
  static constexpr size_t ring = 0;
  static constexpr size_t merge_o = ring + size_t(kStages) * kStageBytes;                // [4][8][128] f32 (8 heads a round)
  static constexpr size_t merge_ml = merge_o + size_t(kConsumerWarps) * kRowG * kD * 4;  // [4][16][2] f32
  static constexpr size_t cands = merge_ml + size_t(kConsumerWarps) * kMaxG * 2 * 4;    // [4][256] u32 + i32
  static constexpr size_t bars = cands + size_t(kConsumerWarps) * kWarpCands * 8;        // 2 x kStages u64
  static constexpr size_t seqS = bars + 2 * kStages * 8;                                 // [kMaxBatch] i32
  static constexpr size_t seqPref = seqS + size_t(kMaxBatch) * 4;                        // [kMaxBatch+1] i64
  static constexpr size_t stats = seqPref + size_t(kMaxBatch + 1) * 8;                   // [16][2] f32
  static constexpr size_t owners = stats + kMaxG * 2 * 4;                                // [kMaxOwners+1] i32
  static constexpr size_t sig = owners + (kMaxOwners + 1) * 4;                           // i32: segment completed its pair
  static constexpr size_t sigseqs = sig + 16;                                            // [kMaxBatch/32] u32 bitmap
  static constexpr size_t total = sigseqs + kMaxBatch / 8;
};
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
  float* logits;   // log2-domain logits [B][Hq][max_len]: the probs buffer, else workspace
  float* probs;    // output probabilities or null (aliases logits when given)
  float* cum;      // H2O score [B][Hkv][max_len] or null
  uint32_t* link_hint;   // H2O candidate hand-off (h2o_link.cuh), all null when not linked
  uint32_t* link_count;
  uint32_t* link_key;
  int32_t* link_pos;
  void* out;
  float* part;     // [slots][kPartFloats]
  unsigned* fin;   // CTAs past the append (status area); the last one publishes the lengths
  unsigned* pair_k;     // [B*Hkv] owners whose K pass is done: their (m, l) are written
  unsigned* pair_v;     // [B*Hkv] owners whose V pass is done: their O is written
  unsigned* pair_done;  // [B*Hkv] (unused)
  float* oacc;          // [B][Hq][128] fp32: the owners' normalised partial O, summed (zero between calls)
  // per-step top-k block signal (all null / 0 when off)
  float* bmass;         // [B*Hkv][bpages]: each page's attention mass from one kv head's group
  float* bsum;          // [B][bpages]: summed over the kv heads (the caller's mass_out, else workspace)
  uint32_t* bkeys;      // [B][bpages]: their order keys
  unsigned* seq_done;   // [B]: pairs finished (the last runs the sequence's top-k)
  float* sig_score;     // [num_pages]
  int32_t* sig_step;    // [num_pages]
  int32_t* sig_topk;    // [B][sig_k] or null
  int sig_k, sig_stepv, bpages;
  int* status;
  int B, max_pages, Hq, Hkv, G, num_pages, max_len, out_f32;
  int page_shift;  // log2(page_size / 16): a pool page holds 1 << page_shift 16-token tiles
  int vec2;        // logit and score rows are 8-byte aligned: key pairs move as float2
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

// Bounded spin of one thread until *word == target: 2^25 sleeps of ~64 ns
// (a few seconds) unless the workspace sets another limit.  On expiry it
// records KVSEL_ERR_TIMEOUT and returns false; the caller carries on with
// whatever the partial slots hold (every index it uses comes from the work
// split, never from those values), so results are unspecified but every
// access stays in bounds and nothing hangs.
__device__ __forceinline__ bool wait_word(const unsigned* word, unsigned target, int* status) {
  const unsigned limit = spin_limit(status, 1u << 25);
  unsigned spins = 0;
  while (*reinterpret_cast<const volatile unsigned*>(word) != target) {
    __nanosleep(64);
    if (++spins >= limit) {
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

// The CTAs owning units [pfirst, plast] of a pair, in order: the owner of
// pfirst, then the owner of the unit right after each owner's range.  Written
// to own[0..n-1], n to own[kMaxOwners]; one thread.
__device__ __forceinline__ int list_owners(int* own, long long pfirst, long long plast, long long U, int NC) {
  int no = 0;
  for (int cc = cta_of(pfirst, U, NC); cc >= 0 && no < kMaxOwners; ++no) {
    own[no] = cc;
    const long long nu = U * (cc + 1) / NC;
    cc = nu > plast ? -1 : cta_of(nu, U, NC);
  }
  own[kMaxOwners] = no;
  return no;
}

// Merge of two (max, sum of exp2) pairs.
__device__ __forceinline__ void ml_merge(float& m, float& l, float mo, float lo) {
  const float mn = fmaxf(m, mo);
  l = mn == -INFINITY ? 0.f : l * exp2f(m - mn) + lo * exp2f(mo - mn);
  m = mn;
}

// A consumer warp's H2O candidates (slots whose new score key is >= the
// row's last threshold), staged in shared memory and handed to the row's
// list with one global atomic per flush.
struct WarpCands {
  uint32_t* key;  // [kWarpCands]
  int32_t* pos;   // [kWarpCands]
  uint32_t n;     // staged entries (warp-uniform)
};

// Every lane offers slot j with new score v (where on).
__device__ __forceinline__ void cands_stage(WarpCands& wc, bool on, int j, float v, uint32_t hk, int lane) {
  const uint32_t k = order_key(v);
  const bool h = on && k >= hk;
  const uint32_t bal = __ballot_sync(0xffffffffu, h);
  if (h) {
    const uint32_t o = wc.n + __popc(bal & ((1u << lane) - 1u));
    wc.key[o] = k;
    wc.pos[o] = j;
  }
  wc.n += __popc(bal);
}

__device__ __forceinline__ void cands_flush(WarpCands& wc, const StepParams& P, int pair, int lane) {
  if (wc.n == 0) return;
  __syncwarp();
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(P.link_count + pair, wc.n);
  base = __shfl_sync(0xffffffffu, base, 0);
  uint32_t* gk = P.link_key + size_t(pair) * kLinkCap;
  int32_t* gp = P.link_pos + size_t(pair) * kLinkCap;
  for (uint32_t i = lane; i < wc.n && base + i < uint32_t(kLinkCap); i += 32) {
    gk[base + i] = wc.key[i];
    gp[base + i] = wc.pos[i];
  }
  __syncwarp();
  wc.n = 0;
}

// Two key pairs of one row: keys k0, k0 + 1 and k2, k2 + 1 of a page starting
// at row[key0]; entries at or past `valid` read as `fill`.
__device__ __forceinline__ float4 load_keys(const float* row, int key0, int valid, int k0, int k2, bool vec2,
                                            float fill) {
  float4 r = make_float4(fill, fill, fill, fill);
  const float* p = row + key0;
  if (vec2 && valid >= kPage) {
    const float2 a = __ldcg(reinterpret_cast<const float2*>(p + k0));
    const float2 b = __ldcg(reinterpret_cast<const float2*>(p + k2));
    r = make_float4(a.x, a.y, b.x, b.y);
  } else {
    if (k0 < valid) r.x = __ldcg(p + k0);
    if (k0 + 1 < valid) r.y = __ldcg(p + k0 + 1);
    if (k2 < valid) r.z = __ldcg(p + k2);
    if (k2 + 1 < valid) r.w = __ldcg(p + k2 + 1);
  }
  return r;
}
__device__ __forceinline__ void st_hint(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st2_hint(float* p, float a, float b, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(a), "f"(b), "l"(pol) : "memory");
}
// Stores key pairs like load_keys reads them, with L2 eviction policy pol.
__device__ __forceinline__ void store_keys(float* row, int key0, int valid, int k0, int k2, bool vec2, float4 v,
                                           uint64_t pol) {
  float* p = row + key0;
  if (vec2 && valid >= kPage) {
    st2_hint(p + k0, v.x, v.y, pol);
    st2_hint(p + k2, v.z, v.w, pol);
  } else {
    if (k0 < valid) st_hint(p + k0, v.x, pol);
    if (k0 + 1 < valid) st_hint(p + k0 + 1, v.y, pol);
    if (k2 < valid) st_hint(p + k2, v.z, pol);
    if (k2 + 1 < valid) st_hint(p + k2 + 1, v.w, pol);
  }
}
// 2^x by the hardware approximation (relative error ~2^-22; -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Per-step top-k block signal of one sequence, run by the CTA that finishes
// the sequence's last (sequence, kv head) pair, all kThreads threads:
//   mass[p]  = the page's attention mass summed over the kv heads (fixed order)
//   chosen   = the sig_k pages of largest mass, ties to the lower page (every
//              page when there are no more), in ascending order: a radix select
//              of the k-th key (four 8-bit digits, most significant first) and
//              an ordered emission by block scans
//   for each chosen page: score[phys] += mass, step[phys] = the step.
// `sm` is shared scratch of sm_words >= 320 words (the ring, free by then);
// the page keys live there too when they fit.
__device__ __forceinline__ uint32_t sig_block_scan(uint32_t v, uint32_t* wt, uint32_t& total) {
  constexpr int kW = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wt[warp] = x;
  __syncthreads();
  uint32_t before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const uint32_t t = wt[w];
    if (w < warp) before += t;
    total += t;
  }
  __syncthreads();
  return before + x - v;
}

__device__ __noinline__ void block_signal(const StepParams& P, int b, int S, uint32_t* sm, int sm_words) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = (S + kPage - 1) / kPage;
  const int k = min(P.sig_k, n);
  float* msum = P.bsum + size_t(b) * P.bpages;
  uint32_t* hist = sm;        // [256]
  uint32_t* wt = sm + 256;    // [32]
  uint32_t* bc = sm + 288;    // [2]: digit, remaining
  // the keys stay in shared memory when they fit (n <= ~16K pages), else in the workspace
  uint32_t* keys = n <= sm_words - 320 ? sm + 320 : P.bkeys + size_t(b) * P.bpages;
  {
    const float* bmb = P.bmass + size_t(b) * P.Hkv * P.bpages;
    constexpr int kU = 4;  // pages per thread in flight, every kv head's load issued before the sums
    for (int p0 = tid; p0 < n; p0 += kU * kThreads) {
      float m[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) m[u] = 0.f;
#pragma unroll 4
      for (int h = 0; h < P.Hkv; ++h) {
        float x[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int p = p0 + u * kThreads;
          x[u] = p < n ? __ldcg(bmb + size_t(h) * P.bpages + p) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) m[u] += x[u];
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int p = p0 + u * kThreads;
        if (p < n) {
          msum[p] = m[u];
          keys[p] = order_key(m[u]);
        }
      }
    }
  }
  __syncthreads();  // the block's own stores, read back below
  uint32_t prefix = 0u, mask = 0u, remaining = uint32_t(k);
  if (k < n) {
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kThreads) hist[i] = 0u;
      __syncthreads();
      for (int p = tid; p < n; p += kThreads) {
        const uint32_t key = keys[p];
        if ((key & mask) == prefix) atomicAdd(hist + ((key >> shift) & 255u), 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits 255 - 8l - j, j = 0..7: counts from the top down
        uint32_t c[8], tot = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - 8 * lane - j];
          tot += c[j];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t above = incl - tot;  // keys with a higher digit than this lane's
        if (above < remaining && remaining <= above + tot) {
          uint32_t cum = above;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (cum < remaining && remaining <= cum + c[j]) {
              bc[0] = uint32_t(255 - 8 * lane - j);
              bc[1] = remaining - cum;
            }
            cum += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= bc[0] << shift;
      mask |= 0xFFu << shift;
      remaining = bc[1];
      __syncthreads();
    }
  }
  // ordered emission: every key above T, then the first `remaining` equal to T
  const uint32_t T = prefix;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  int32_t* tko = P.sig_topk ? P.sig_topk + size_t(b) * P.sig_k : nullptr;
  uint32_t out_base = 0u, eq_base = 0u;
#pragma unroll 1
  for (int c0 = 0; c0 < n; c0 += kThreads * 8) {
    uint32_t kk[8];
    uint32_t neq = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = c0 + 8 * tid + j;
      kk[j] = p < n ? keys[p] : 0u;
      if (p < n && k < n && kk[j] == T) ++neq;
    }
    uint32_t eq_tot;
    uint32_t eq_rank = eq_base + sig_block_scan(neq, wt, eq_tot);
    bool take[8];
    uint32_t ntake = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = c0 + 8 * tid + j;
      bool t = false;
      if (p < n) {
        if (k == n || kk[j] > T) t = true;
        else if (kk[j] == T) t = eq_rank++ < remaining;
      }
      take[j] = t;
      ntake += t ? 1u : 0u;
    }
    uint32_t out_tot;
    uint32_t o = out_base + sig_block_scan(ntake, wt, out_tot);
    // the taken pages' block-table entries, masses and old scores, all loads issued together
    int phys[8];
    float ms[8], old[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = c0 + 8 * tid + j;
      phys[j] = take[j] ? __ldcg(bt + p) : -1;
      ms[j] = take[j] ? __ldcg(msum + p) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (take[j] && unsigned(phys[j]) >= unsigned(P.num_pages)) {
        report(P.status, KVSEL_ERR_BAD_INDEX);
        take[j] = false;
      }
      old[j] = take[j] ? __ldcg(P.sig_score + phys[j]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!take[j]) continue;
      if (tko) tko[o] = c0 + 8 * tid + j;
      P.sig_score[phys[j]] = old[j] + ms[j];
      P.sig_step[phys[j]] = P.sig_stepv;
      ++o;
    }
    out_base += out_tot;
    eq_base += eq_tot;
  }
  if (tko)
    for (int i = k + tid; i < P.sig_k; i += kThreads) tko[i] = -1;
}

// kSig: the per-step block signal is on (P.bmass and the rest set); the
// default instantiation carries none of its code.  kWide: more than 8 q
// heads per kv head (up to 16).
template <bool kSig, bool kWide>
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
  int& sLastPair = *reinterpret_cast<int*>(smem + SmemLayout::sig);  // this segment completed its pair
  uint32_t* sSigSeqs = reinterpret_cast<uint32_t*>(smem + SmemLayout::sigseqs);  // [kMaxBatch / 32]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = gridDim.x, c = blockIdx.x;
  const bool append = P.k_new != nullptr;
  const int Hkv = P.Hkv, G = P.G;

  // ---- lengths, unit prefix, this CTA's range ----
  // Lengths, positions and the block table are read before this kernel waits
  // for the previous one (see the K pass end), so they are read from L2, which
  // holds every completed kernel's writes (a compaction that precedes this
  // launch lets it start only once it has completed).
  for (int b = tid; b < P.B; b += kThreads) sS[b] = __ldcg(P.seq_lens + b) + (append ? 1 : 0);
  __syncthreads();
  if (tid == 0) {
    long long acc = 0;
    int bad = 0;
    for (int b = 0; b < P.B; ++b) {
      sPref[b] = acc;
      const int S = sS[b];
      const int np = (S + kPage - 1) / kPage;
      if (S < (append ? 1 : 0) || S > P.max_len || np > (P.max_pages << P.page_shift)) bad = 1;
      acc += (long long)Hkv * np;
    }
    sPref[P.B] = bad ? -1 : acc;
  }
  for (int i = tid; i < kMaxBatch / 32; i += kThreads) sSigSeqs[i] = 0u;
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
        const int phys = __ldcg(P.block_table + size_t(b) * P.max_pages + (S_old >> (4 + P.page_shift)));
        if (unsigned(phys) < unsigned(P.num_pages)) {
          const int psz = kPage << P.page_shift;
          const size_t row = (size_t(phys) * Hkv + kvh) * psz + (S_old & (psz - 1));
          const int t = tid & 15;
          const __nv_bfloat16* src = (tid < 16 ? P.k_new : P.v_new) + (size_t(b) * Hkv + kvh) * kD;
          __nv_bfloat16* dst = (tid < 16 ? P.k_pool : P.v_pool) + row * kD;
          reinterpret_cast<uint4*>(dst)[t] = reinterpret_cast<const uint4*>(src)[t];
        } else if (tid == 0) {
          report(P.status, KVSEL_ERR_BAD_INDEX);
        }
        if (tid == 0 && P.pos_map)
          P.pos_map[(size_t(b) * Hkv + kvh) * P.max_len + S_old] = P.next_pos ? __ldcg(P.next_pos + b) : S_old;
      }
    }
    fence_proxy_async_global();
  }
  __syncthreads();
  // Every CTA has read the old lengths and positions (and appended) once all
  // have counted themselves here: the last one publishes the new ones, long
  // before a kernel launched after this one can start.  (A preceding H2O
  // select reads the lengths before it lets this launch start.)
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

  const int n = int(u1 - u0);       // pages of the range
  const int nsk = (n + 1) >> 1;     // stages per pass
  const int g = lane >> 2, qd = lane & 3;
  const bool head_ok = g < G;
  const bool head_ok2 = kWide && g + kRowG < G;  // rows 8..15 carry head g + 8
  const bool vec2 = P.vec2 != 0;
  const int k0 = 2 * qd, k2 = 8 + 2 * qd;  // this lane's keys in a page: k0, k0+1, k2, k2+1

  // Stage t of a pass holds the pass's pages 2t and 2t + 1; the K pass uses
  // ring stages 0 .. nsk-1, the V pass nsk .. 2 nsk - 1.  Ring stage r
  // belongs to consumer warp r % 4.
  auto first_page = [&](int i, int base) -> int {  // this warp's first page >= i
    const int t = i >> 1;
    const int tt = t + ((warp - (base + t) % kConsumerWarps) + kConsumerWarps) % kConsumerWarps;
    return tt == t ? i : 2 * tt;
  };
  auto next_page = [](int i) -> int { return (i & 1) ? i + 2 * kConsumerWarps - 1 : i + 1; };

  if (warp >= kConsumerWarps) {
    // ================= producers =================
    // Producer warp pw fills the stages t with t % kProducerWarps == pw.
    // Every lane resolves one page of a 32-page chunk (block table entry ->
    // TMA row coordinate), two chunks ahead of use, so the dependent
    // block-table loads never sit between two TMA issues.
    const int pw = warp - kConsumerWarps;
    if (n > 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto resolve = [&](int i) -> int {  // TMA row of CTA-local page i (or -1 past the end)
        if (i >= n) return -1;
        int b, kvh, pg;
        loc.locate(u0 + i, b, kvh, pg);
        int phys = __ldcg(P.block_table + size_t(b) * P.max_pages + (pg >> P.page_shift));
        if (unsigned(phys) >= unsigned(P.num_pages)) {
          report(P.status, KVSEL_ERR_BAD_INDEX);
          phys = 0;
        }
        // the 16-token tile pg of a page of 16 << page_shift rows
        return ((phys * Hkv + kvh) << P.page_shift | (pg & ((1 << P.page_shift) - 1))) * kPage;
      };
      bool stop = false;
#pragma unroll 1
      for (int pass = 0; pass < 2 && !stop; ++pass) {
        const CUtensorMap* tm = pass ? &tmV : &tmK;
        int y_cur = resolve(lane);
        int y_next = resolve(32 + lane);
#pragma unroll 1
        for (int i0 = 0; i0 < n && !stop; i0 += 32) {
          const int y_after = resolve(i0 + 64 + lane);  // issued early; used two chunks later
#pragma unroll 1
          for (int k = 0; k < 32 && i0 + k < n; k += 2) {
            const int t = pass * nsk + ((i0 + k) >> 1);
            if (t % kProducerWarps != pw) continue;  // the other producer's stage
            const int ya = __shfl_sync(0xffffffffu, y_cur, k);
            const int yb = __shfl_sync(0xffffffffu, y_cur, k + 1);
            const bool two = i0 + k + 1 < n;
            const int s = t % kStages;
            bool ok = true;
            if (t >= kStages) ok = mbar_wait(smem_u32(&empty[s]), ((t / kStages) + 1) & 1, P.status);
            if (!__all_sync(0xffffffffu, ok)) {
              stop = true;
              break;
            }
            if (lane == 0) {
              const uint32_t dst = smem_u32(smem + SmemLayout::ring + s * kStageBytes);
              const uint32_t bar = smem_u32(&full[s]);
              mbar_expect_tx(bar, two ? kStageBytes : kPageBytes);
              tma_load_3d(dst, tm, 0, ya, 0, bar, pol);
              if (two) tma_load_3d(dst + kPageBytes, tm, 0, yb, 0, bar, pol);
            }
            __syncwarp();
          }
          y_cur = y_next;
          y_next = y_after;
        }
      }
    }
  } else {
    const int mi = lane >> 3, r8 = lane & 7;
    bool alive = true;  // false once a ring wait ran out: the warp then leaves the ring alone
    const uint64_t keep_l2 = l2_policy_evict_last(), drop_l2 = l2_policy_evict_first();

    // ================= K pass =================
#pragma unroll 1
    for (long long u = u0; u < u1;) {
      int b, kvh, pg;
      loc.locate(u, b, kvh, pg);
      const int S = sS[b];
      const int np = loc.pages(b);
      const long long seg_end = min(u1, u + (np - pg));
      const int pair = b * Hkv + kvh;

      // A rows: head g in rows 0..7; with more than 8 heads, head g + 8 in rows 8..15
      uint32_t qa[8][2], qb[8][2];
      {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            P.q + (size_t(b) * P.Hq + kvh * G + (head_ok ? g : 0)) * kD);
        const uint32_t* qrow2 = reinterpret_cast<const uint32_t*>(
            P.q + (size_t(b) * P.Hq + kvh * G + (head_ok2 ? g + kRowG : 0)) * kD);
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          qa[kt][0] = head_ok ? qrow[(16 * kt + 2 * qd) >> 1] : 0u;
          qa[kt][1] = head_ok ? qrow[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
          qb[kt][0] = head_ok2 ? qrow2[(16 * kt + 2 * qd) >> 1] : 0u;
          qb[kt][1] = head_ok2 ? qrow2[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
        }
      }
      float* lrow = head_ok ? P.logits + (size_t(b) * P.Hq + kvh * G + g) * P.max_len : nullptr;
      float* lrow2 = head_ok2 ? P.logits + (size_t(b) * P.Hq + kvh * G + g + kRowG) * P.max_len : nullptr;
      float m_l = -INFINITY, l_l = 0.f;    // this lane's keys of the segment, head g
      float m_l2 = -INFINITY, l_l2 = 0.f;  // head g + 8

      const int i_begin = int(u - u0), i_end = int(seg_end - u0);
#pragma unroll 1
      for (int i = first_page(i_begin, 0); i < i_end && alive; i = next_page(i)) {
        const int t = i >> 1, s = t % kStages;
        if (!mbar_wait(smem_u32(&full[s]), (t / kStages) & 1, P.status)) {
          alive = false;
          break;
        }
        const uint32_t kb = smem_u32(smem + SmemLayout::ring + s * kStageBytes + (i & 1) * kPageBytes);
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          const int key = (mi >> 1) * 8 + r8;
          const int uu = 2 * kt + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + tile_off(key, uu), b0, b1, b2, b3);
          mma_bf16_16816(s0, qa[kt][0], qb[kt][0], qa[kt][1], qb[kt][1], b0, b1);
          mma_bf16_16816(s1, qa[kt][0], qb[kt][0], qa[kt][1], qb[kt][1], b2, b3);
        }
        __syncwarp();
        if ((i & 1) || i + 1 == n)  // the stage's last page: its K rows are in registers now
          if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        const int key0 = (pg + (i - i_begin)) * kPage;
        const int valid = S - key0;  // >= 1
        // one head's four logits of the page: stored (read back by the V pass) and folded
        // into the lane's running (max, sum of exp2)
        auto fold = [&](float a, float bq, float cq, float dq, float* row, float& m, float& l) {
          float4 x;
          x.x = k0 < valid ? a * P.scale_log2 : -INFINITY;
          x.y = k0 + 1 < valid ? bq * P.scale_log2 : -INFINITY;
          x.z = k2 < valid ? cq * P.scale_log2 : -INFINITY;
          x.w = k2 + 1 < valid ? dq * P.scale_log2 : -INFINITY;
          if (row) store_keys(row, key0, valid, k0, k2, vec2, x, keep_l2);
          const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
          if (mx != -INFINITY) {
            const float m_new = fmaxf(m, mx);
            l = l * ex2(m - m_new) + ((ex2(x.x - m_new) + ex2(x.y - m_new)) +
                                      (ex2(x.z - m_new) + ex2(x.w - m_new)));
            m = m_new;
          }
        };
        fold(s0[0], s0[1], s1[0], s1[1], lrow, m_l, l_l);
        if (kWide) fold(s0[2], s0[3], s1[2], s1[3], lrow2, m_l2, l_l2);
      }

      // ---- the segment's (m, l) per head: over the head's 4 lanes, then the 4 warps ----
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m_l, off);
        const float lo = __shfl_xor_sync(0xffffffffu, l_l, off);
        ml_merge(m_l, l_l, mo, lo);
        if (kWide) {
          const float mo2 = __shfl_xor_sync(0xffffffffu, m_l2, off);
          const float lo2 = __shfl_xor_sync(0xffffffffu, l_l2, off);
          ml_merge(m_l2, l_l2, mo2, lo2);
        }
      }
      if (qd == 0 && head_ok) {
        wml[(warp * kMaxG + g) * 2 + 0] = m_l;
        wml[(warp * kMaxG + g) * 2 + 1] = l_l;
      }
      if (qd == 0 && head_ok2) {
        wml[(warp * kMaxG + g + kRowG) * 2 + 0] = m_l2;
        wml[(warp * kMaxG + g + kRowG) * 2 + 1] = l_l2;
      }
      consumer_sync();
      if (tid < G) {
        float M = -INFINITY, L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
          ml_merge(M, L, wml[(w * kMaxG + tid) * 2], wml[(w * kMaxG + tid) * 2 + 1]);
        float* slot = P.part + size_t(c + pair) * kPartFloats;
        slot[tid] = M;
        slot[kMaxG + tid] = L;
      }
      __threadfence();  // the slot and this segment's logits
      consumer_sync();
      u = seg_end;
    }

    // The kernel before this one in the stream (an H2O select, when it lets
    // this launch start early) reads the H2O scores and candidate lists that
    // the V pass writes, and writes the thresholds it reads: only the K pass
    // overlaps it.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // announce: this CTA's (m, l) partials (and logits) for its pairs are written
    if (tid == 0) {
      for (long long u = u0; u < u1;) {
        int b, kvh, pg;
        loc.locate(u, b, kvh, pg);
        const int pair = b * Hkv + kvh;
        // the first owner gives the pair a fresh H2O candidate list before anyone can append
        if (P.link_count && pg == 0) P.link_count[pair] = 0u;
        __threadfence();
        atomicAdd(P.pair_k + pair, 1u);
        u = min(u1, u + (loc.pages(b) - pg));
      }
    }

    // ================= V pass =================
    WarpCands wc;
    wc.key = reinterpret_cast<uint32_t*>(smem + SmemLayout::cands) + warp * kWarpCands;
    wc.pos = reinterpret_cast<int32_t*>(smem + SmemLayout::cands + kConsumerWarps * kWarpCands * 4) +
             warp * kWarpCands;
    wc.n = 0;
    // after the head sums below, lanes of even heads hold key kc of each page
    const bool csum_lane = (g & 1) == 0;
    const int kc = ((g & 4) ? k2 : k0) + ((g & 2) ? 1 : 0);
#pragma unroll 1
    for (long long u = u0; u < u1;) {
      int b, kvh, pg;
      loc.locate(u, b, kvh, pg);
      const int S = sS[b];
      const int np = loc.pages(b);
      const long long seg_end = min(u1, u + (np - pg));
      const int pair = b * Hkv + kvh;
      const size_t hrow = (size_t(b) * P.Hq + kvh * G + g) * P.max_len;
      const float* lrow = head_ok ? P.logits + hrow : nullptr;
      float* prow = (head_ok && P.probs) ? P.probs + hrow : nullptr;
      const float* lrow2 = head_ok2 ? P.logits + hrow + size_t(kRowG) * P.max_len : nullptr;  // head g + 8
      float* prow2 = (head_ok2 && P.probs) ? P.probs + hrow + size_t(kRowG) * P.max_len : nullptr;
      float* crow = P.cum ? P.cum + (size_t(b) * Hkv + kvh) * P.max_len : nullptr;
      const bool cown = crow != nullptr && csum_lane;
      // the row's last H2O threshold: collect the slots at or above it (0: no list)
      const uint32_t hk = (crow && P.link_hint) ? __ldcg(P.link_hint + pair) : 0u;

      const int i_begin = int(u - u0), i_end = int(seg_end - u0);
      // the stored logits and old score of one of this warp's pages
      auto fetch = [&](int ii, float4& lg, float4& lg2, float& cs) {
        lg = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        lg2 = lg;
        cs = 0.f;
        if (ii < i_end) {
          const int key0 = (pg + (ii - i_begin)) * kPage;
          const int valid = S - key0;
          if (lrow) lg = load_keys(lrow, key0, valid, k0, k2, vec2, -INFINITY);
          if (kWide && lrow2) lg2 = load_keys(lrow2, key0, valid, k0, k2, vec2, -INFINITY);
          if (cown && kc < valid) cs = __ldcg(crow + key0 + kc);
        }
      };
      int i = first_page(i_begin, nsk);
      float4 lgA, lgB, lgA2, lgB2;
      float csA, csB;
      fetch(i, lgA, lgA2, csA);  // two pages ahead: issued before the wait below
      fetch(next_page(i), lgB, lgB2, csB);
      if (tid == 0) {
        const long long pfirst = sPref[b] + (long long)kvh * np;
        const int no = list_owners(sOwn, pfirst, pfirst + np - 1, U, NC);
        wait_word(P.pair_k + pair, unsigned(no), P.status);  // every owner's (m, l) is written
      }
      consumer_sync();
      const int nown = sOwn[kMaxOwners];
      // the pair's (M, 1/L) per head: warp w merges heads w, w + 4 over the owners, a lane per owner
      for (int gg = warp; gg < G; gg += kConsumerWarps) {
        float m = -INFINITY, l = 0.f;
        for (int k = lane; k < nown; k += 32) {
          const float* sl = P.part + size_t(sOwn[k] + pair) * kPartFloats;
          ml_merge(m, l, __ldcg(sl + gg), __ldcg(sl + kMaxG + gg));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          const float mo = __shfl_xor_sync(0xffffffffu, m, off);
          const float lo = __shfl_xor_sync(0xffffffffu, l, off);
          ml_merge(m, l, mo, lo);
        }
        if (lane == 0) {
          sStat[gg * 2] = m;
          sStat[gg * 2 + 1] = l > 0.f ? 1.f / l : 0.f;
        }
      }
      consumer_sync();
      const float Mg = head_ok ? sStat[g * 2] : 0.f;
      const float Ig = head_ok ? sStat[g * 2 + 1] : 0.f;
      const float Mg2 = head_ok2 ? sStat[(g + kRowG) * 2] : 0.f;
      const float Ig2 = head_ok2 ? sStat[(g + kRowG) * 2 + 1] : 0.f;

      float o[16][4];
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

#pragma unroll 1
      for (; i < i_end && alive; i = next_page(i)) {
        const float4 lg = lgA, lg2 = lgA2;
        const float cs = csA;
        lgA = lgB;
        lgA2 = lgB2;
        csA = csB;
        fetch(next_page(next_page(i)), lgB, lgB2, csB);
        const int t = nsk + (i >> 1), s = t % kStages;
        if (!mbar_wait(smem_u32(&full[s]), (t / kStages) & 1, P.status)) {
          alive = false;
          break;
        }
        const uint32_t vb = smem_u32(smem + SmemLayout::ring + s * kStageBytes + (i & 1) * kPageBytes);
        const int key0 = (pg + (i - i_begin)) * kPage;
        const int valid = S - key0;  // >= 1

        // final probabilities (keys past the length hold -inf: p = 0)
        const float p0 = ex2(lg.x - Mg) * Ig, p1 = ex2(lg.y - Mg) * Ig;
        const float p2 = ex2(lg.z - Mg) * Ig, p3 = ex2(lg.w - Mg) * Ig;
        if (prow) store_keys(prow, key0, valid, k0, k2, vec2, make_float4(p0, p1, p2, p3), drop_l2);
        float p4 = 0.f, p5 = 0.f, p6 = 0.f, p7 = 0.f;  // head g + 8
        if (kWide) {
          p4 = ex2(lg2.x - Mg2) * Ig2;
          p5 = ex2(lg2.y - Mg2) * Ig2;
          p6 = ex2(lg2.z - Mg2) * Ig2;
          p7 = ex2(lg2.w - Mg2) * Ig2;
          if (prow2) store_keys(prow2, key0, valid, k0, k2, vec2, make_float4(p4, p5, p6, p7), drop_l2);
        }
        if (kSig || crow) {
          // the group's probability per key (heads g and g + 8 first added in
          // the lane), a transposing sum over the 8 head rows: lanes of heads
          // with bit 2 set keep keys k2, k2 + 1, the others k0, k0 + 1; bit 1
          // then picks one of the two; bit 0 completes the sum
          const float q0 = p0 + p4, q1 = p1 + p5, q2 = p2 + p6, q3 = p3 + p7;
          const bool hi4 = (g & 4) != 0, hi2 = (g & 2) != 0;
          float a = hi4 ? q2 : q0, bb = hi4 ? q3 : q1;
          a += __shfl_xor_sync(0xffffffffu, hi4 ? q0 : q2, 16);
          bb += __shfl_xor_sync(0xffffffffu, hi4 ? q1 : q3, 16);
          float x = hi2 ? bb : a;
          x += __shfl_xor_sync(0xffffffffu, hi2 ? a : bb, 8);
          x += __shfl_xor_sync(0xffffffffu, x, 4);
          const bool on = cown && kc < valid;
          if (crow) {
            const float nv = ((append && key0 + kc == S - 1) ? 0.f : cs) + x;  // the appended slot starts from zero
            if (on) __stcg(crow + key0 + kc, nv);
            if (hk) cands_stage(wc, on, key0 + kc, nv, hk, lane);
          }
          if (kSig) {  // the page's mass from this group: the 16 keys held by the even-head lanes
            float mass = (csum_lane && kc < valid) ? x : 0.f;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mass += __shfl_xor_sync(0xffffffffu, mass, off);
            if (lane == 0) P.bmass[size_t(pair) * P.bpages + key0 / kPage] = mass;
          }
        }

        // O += P V with P as a bf16 high part plus its bf16 residual.  Up to 8 heads: the
        // high parts in rows 0..7, the residuals in rows 8..15, one MMA.  More than 8: heads
        // g and g + 8 in rows g and g + 8, one MMA for the high parts and one for the residuals
        // into the same accumulators.
        const uint32_t hi01 = pack_bf16x2(p0, p1);
        const uint32_t hi23 = pack_bf16x2(p2, p3);
        const uint32_t lo01 = pack_bf16x2(p0 - bf16lo_to_f32(hi01), p1 - bf16hi_to_f32(hi01));
        const uint32_t lo23 = pack_bf16x2(p2 - bf16lo_to_f32(hi23), p3 - bf16hi_to_f32(hi23));
        uint32_t hi45 = 0u, hi67 = 0u, lo45 = 0u, lo67 = 0u;
        if (kWide) {
          hi45 = pack_bf16x2(p4, p5);
          hi67 = pack_bf16x2(p6, p7);
          lo45 = pack_bf16x2(p4 - bf16lo_to_f32(hi45), p5 - bf16hi_to_f32(hi45));
          lo67 = pack_bf16x2(p6 - bf16lo_to_f32(hi67), p7 - bf16hi_to_f32(hi67));
        }
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
          if (kWide) {
            mma_bf16_16816(o[2 * j], hi01, hi45, hi23, hi67, b0, b1);
            mma_bf16_16816(o[2 * j + 1], hi01, hi45, hi23, hi67, b2, b3);
            mma_bf16_16816(o[2 * j], lo01, lo45, lo23, lo67, b0, b1);
            mma_bf16_16816(o[2 * j + 1], lo01, lo45, lo23, lo67, b2, b3);
          } else {
            mma_bf16_16816(o[2 * j], hi01, lo01, hi23, lo23, b0, b1);
            mma_bf16_16816(o[2 * j + 1], hi01, lo01, hi23, lo23, b2, b3);
          }
        }
        __syncwarp();
        if ((i & 1) || i + 1 == n)
          if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (hk && wc.n > uint32_t(kWarpCands - 16)) cands_flush(wc, P, pair, lane);
      }
      if (hk) cands_flush(wc, P, pair, lane);

      // ---- the segment's O (already normalised): the 4 warps' sum, added into the pair's fp32
      // accumulator; the pair's last owner to get here writes O and clears the accumulator, so
      // no owner waits for the others ----
      // (eight heads a round through the shared buffer: heads 0..7, then 8..15 when the group
      // is wider)
      float* oacc = P.oacc + (size_t(b) * P.Hq + kvh * G) * kD;
#pragma unroll 1
      for (int half = 0; half < (kWide ? 2 : 1); ++half) {
        const int gh = half * kRowG, hn = min(kRowG, G - gh);  // this merge pass's first head, heads
        if (g < hn) {
          float* dst = wo + (warp * kRowG + g) * kD;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
            *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) =
                kWide ? (half ? make_float2(o[nt][2], o[nt][3]) : make_float2(o[nt][0], o[nt][1]))
                      : make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
        }
        consumer_sync();
        for (int idx = tid; idx < hn * kD; idx += kConsumerWarps * 32)
          atomicAdd(oacc + gh * kD + idx,
                    ((wo[idx] + wo[kRowG * kD + idx]) + wo[2 * kRowG * kD + idx]) + wo[3 * kRowG * kD + idx]);
        if (kWide && half == 0) consumer_sync();  // the next round overwrites the buffer
      }
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        const int no = sOwn[kMaxOwners];  // this segment's owners (listed at its start)
        const int last = atomicAdd(P.pair_v + pair, 1u) + 1u == unsigned(no);
        if (last) {
          __threadfence();
          P.pair_k[pair] = 0u;
          P.pair_v[pair] = 0u;
          if (kSig) {  // every owner's page masses are written too: count the pair for its sequence
            if (atomicAdd(P.seq_done + b, 1u) + 1u == unsigned(Hkv)) {
              P.seq_done[b] = 0u;
              __threadfence();
              atomicOr(sSigSeqs + (b >> 5), 1u << (b & 31));  // run after the V pass (it needs the ring)
            }
          }
        }
        sLastPair = last;
      }
      consumer_sync();
      if (sLastPair) {
        for (int idx = tid; idx < G * kD; idx += kConsumerWarps * 32) {
          const float v = __ldcg(oacc + idx);
          __stcg(oacc + idx, 0.f);
          const size_t oi = (size_t(b) * P.Hq + kvh * G) * kD + idx;
          if (P.out_f32) static_cast<float*>(P.out)[oi] = v;
          else static_cast<__nv_bfloat16*>(P.out)[oi] = __float2bfloat16_rn(v);
        }
      }
      u = seg_end;
    }
  }

  // ================= zero-length sequences, block signals =================
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (c == 0) {
    for (int b = 0; b < P.B; ++b)  // sequences without keys: O = 0 (and no block signal)
      if (sS[b] == 0) {
        for (int idx = tid; idx < P.Hq * kD; idx += kThreads) {
          const size_t oi = size_t(b) * P.Hq * kD + idx;
          if (P.out_f32) static_cast<float*>(P.out)[oi] = 0.f;
          else static_cast<__nv_bfloat16*>(P.out)[oi] = __float2bfloat16_rn(0.f);
        }
        if (P.sig_topk)
          for (int i = tid; i < P.sig_k; i += kThreads) P.sig_topk[size_t(b) * P.sig_k + i] = -1;
      }
  }
  if (kSig) {  // the block signal of every sequence whose last pair this CTA completed
    __syncthreads();
    for (int w = 0; w < (P.B + 31) / 32; ++w) {
      uint32_t bits = sSigSeqs[w];
      while (bits) {
        const int b = w * 32 + __ffs(bits) - 1;
        bits &= bits - 1;
        block_signal(P, b, sS[b], reinterpret_cast<uint32_t*>(smem + SmemLayout::ring),
                     int((size_t(kStages) * kStageBytes) / 4));
        __syncthreads();
      }
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
  size_t pair_off, oacc_off, part_off, logit_off, sig_off, total;
};

// The finish counter lives in the workspace's status area (byte 64); the
// three per-pair readiness counters follow it, then the fp32 O accumulator.
// Everything before part_off must be zero when a call starts; each call leaves
// it so.
DecodeWs decode_ws_layout(int batch, int Hkv, int Hq, int max_len, bool with_probs) {
  DecodeWs w;
  size_t off = kStatusBytes;
  w.pair_off = off;
  off = align_up(off + size_t(batch) * Hkv * 3 * sizeof(unsigned), 256);
  w.oacc_off = off;
  off = align_up(off + size_t(batch) * Hq * kD * sizeof(float), 256);
  w.part_off = off;
  off = align_up(off + (size_t(kMaxCtas) + size_t(batch) * Hkv) * kPartFloats * sizeof(float), 256);
  w.logit_off = off;
  if (!with_probs) off = align_up(off + size_t(batch) * Hq * max_len * sizeof(float), 256);
  w.sig_off = off;  // block-signal scratch follows (decode_sig_bytes)
  w.total = off;
  return w;
}

// Block-signal scratch: sequence counters [B], per-group page masses
// [B*Hkv][bpages], summed masses [B][bpages] and their keys [B][bpages].
size_t decode_sig_bytes(int batch, int Hkv, int max_len) {
  const size_t bp = size_t((max_len + kPage - 1) / kPage);
  return align_up(size_t(batch) * 4, 256) + align_up(size_t(batch) * Hkv * bp * 4, 256) +
         2 * align_up(size_t(batch) * bp * 4, 256);
}

// Co-resident CTAs per SM of the kernel instantiation (the launch sizes its
// grid from it); sets the shared-memory attribute on first use.
template <bool kSig, bool kWide>
int ctas_per_sm() {
  static int cached = 0;
  if (cached) return cached;
  if (cudaFuncSetAttribute(decode_step_kernel<kSig, kWide>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemBytes)) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_step_kernel<kSig, kWide>, kThreads, kSmemBytes) !=
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

extern "C" size_t kvsel_decode_attn_ex_workspace(const kvsel_paged_kv* kv, int batch, int max_len, int with_probs,
                                                 int with_signal) {
  const size_t base = kvsel_decode_attn_workspace(kv, batch, max_len, with_probs);
  if (!base || !with_signal) return base;
  return base + decode_sig_bytes(batch, kv->num_kv_heads, max_len);
}

extern "C" kvsel_status kvsel_decode_attn(const kvsel_paged_kv* kv, const int32_t* block_table,
                                          int max_pages, int32_t* seq_lens, int batch, const void* q,
                                          const void* k_new, const void* v_new, int32_t* pos_map,
                                          int32_t* next_pos, float scale, void* out, int out_dtype,
                                          float* probs, float* h2o_cum, int max_len, int num_ctas,
                                          void* workspace, size_t ws_bytes, void* h2o_link,
                                          size_t h2o_link_bytes, void* stream) {
  return kvsel_decode_attn_ex(kv, block_table, max_pages, seq_lens, batch, q, k_new, v_new, pos_map, next_pos,
                              scale, out, out_dtype, probs, h2o_cum, max_len, num_ctas, nullptr, workspace,
                              ws_bytes, h2o_link, h2o_link_bytes, stream);
}

extern "C" kvsel_status kvsel_decode_attn_ex(const kvsel_paged_kv* kv, const int32_t* block_table,
                                             int max_pages, int32_t* seq_lens, int batch, const void* q,
                                             const void* k_new, const void* v_new, int32_t* pos_map,
                                             int32_t* next_pos, float scale, void* out, int out_dtype,
                                             float* probs, float* h2o_cum, int max_len, int num_ctas,
                                             const kvsel_block_signal* signal, void* workspace, size_t ws_bytes,
                                             void* h2o_link, size_t h2o_link_bytes, void* stream) {
  const std::string fn = "kvsel_decode_attn: ";
  if (!kv || !kv->k_pool || !kv->v_pool)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv pools must be non-NULL");
  if (kv->head_dim != kD || page_shift_of(kv->page_size) < 0)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16, 32, 64, 128 or 256 are implemented");
  if (signal && kv->page_size != kPage)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "the block signal is implemented for page_size 16 only");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (G > kMaxG) return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 16 q heads per kv head are implemented");
  if (kv->num_pages < 1 || (long long)kv->num_pages * Hkv * kv->page_size >= (1LL << 31))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_pages * num_kv_heads * page_size must be in [1, 2^31)");
  if ((long long)max_pages << page_shift_of(kv->page_size) >= (1LL << 31))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "max_pages * page_size / 16 must be below 2^31");
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
  if (signal) {
    if (signal->topk_blocks < 1 || !signal->block_score || !signal->block_step)
      return fail(KVSEL_ERR_INVALID_ARG, fn + "block signal: topk_blocks >= 1, block_score and block_step required");
  }
  const size_t need = L.total + (signal ? decode_sig_bytes(batch, Hkv, max_len) : 0);
  if (ws_bytes < need)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(need));
  if (!aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace must be 256-byte aligned");
  if (h2o_link && (!aligned(h2o_link, 256) || h2o_link_bytes < link_bytes(batch * Hkv)))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "h2o_link must be a 256-byte aligned H2O evict workspace of at least " +
                                           std::to_string(link_bytes(batch * Hkv)) + " bytes");

  const bool wide = G > kRowG;
  const int occ = signal ? (wide ? ctas_per_sm<true, true>() : ctas_per_sm<true, false>())
                         : (wide ? ctas_per_sm<false, true>() : ctas_per_sm<false, false>());
  if (occ < 1) return fail(KVSEL_ERR_CUDA, fn + "cannot configure the decode kernel (occupancy 0)");
  const int resident = sm_count() * occ;
  const int nc = num_ctas == 0 ? std::min(resident, kMaxCtas) : num_ctas;
  if (nc > resident)
    return fail(KVSEL_ERR_INVALID_ARG,
                fn + "num_ctas exceeds the co-resident CTA count " + std::to_string(resident));

  CUtensorMap tmK, tmV;
  const uint64_t rows = uint64_t(kv->num_pages) * Hkv * kv->page_size;
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
  P.logits = probs ? probs : reinterpret_cast<float*>(ws + L.logit_off);
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
  P.pair_k = reinterpret_cast<unsigned*>(ws + L.pair_off);
  P.pair_v = P.pair_k + size_t(batch) * Hkv;
  P.pair_done = P.pair_v + size_t(batch) * Hkv;
  P.oacc = reinterpret_cast<float*>(ws + L.oacc_off);
  P.status = reinterpret_cast<int*>(ws);
  P.B = batch;
  P.max_pages = max_pages;
  P.page_shift = page_shift_of(kv->page_size);
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.num_pages = kv->num_pages;
  P.max_len = max_len;
  P.out_f32 = out_dtype == KVSEL_F32;
  P.vec2 = (max_len % 2 == 0) && aligned(P.logits, 8) && (!h2o_cum || aligned(h2o_cum, 8));
  P.bpages = (max_len + kPage - 1) / kPage;
  P.bmass = P.bsum = nullptr;
  P.bkeys = nullptr;
  P.seq_done = nullptr;
  P.sig_score = nullptr;
  P.sig_step = P.sig_topk = nullptr;
  P.sig_k = P.sig_stepv = 0;
  if (signal) {
    const size_t bp = size_t(P.bpages);
    size_t off = L.sig_off;
    P.seq_done = reinterpret_cast<unsigned*>(ws + off);
    off += align_up(size_t(batch) * 4, 256);
    P.bmass = reinterpret_cast<float*>(ws + off);
    off += align_up(size_t(batch) * Hkv * bp * 4, 256);
    P.bsum = signal->mass_out ? signal->mass_out : reinterpret_cast<float*>(ws + off);
    off += align_up(size_t(batch) * bp * 4, 256);
    P.bkeys = reinterpret_cast<uint32_t*>(ws + off);
    P.sig_score = signal->block_score;
    P.sig_step = signal->block_step;
    P.sig_topk = signal->topk_out;
    P.sig_k = signal->topk_blocks;
    P.sig_stepv = signal->step;
  }
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  // No cooperative attribute: that would hold the launch until the whole grid
  // fits at once.  The grid is at most the co-resident CTA count, and its
  // cross-CTA waits come after the K pass, when every CTA is resident.  The
  // launch may start while the previous kernel runs if that kernel allows it
  // (the H2O select does); the kernel waits for it before its V pass.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before("decode_step", st);
  const cudaError_t e =
      signal ? (wide ? cudaLaunchKernelEx(&cfg, decode_step_kernel<true, true>, tmK, tmV, P)
                     : cudaLaunchKernelEx(&cfg, decode_step_kernel<true, false>, tmK, tmV, P))
             : (wide ? cudaLaunchKernelEx(&cfg, decode_step_kernel<false, true>, tmK, tmV, P)
                     : cudaLaunchKernelEx(&cfg, decode_step_kernel<false, false>, tmK, tmV, P));
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
