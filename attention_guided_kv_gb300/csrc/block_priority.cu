// Block offload priority from per-token attention scores (sm_103a).
//
// What it computes ("Sparse attention x KV-cache offloading: eight
// questions" §2.1, §3.1, §3.2, §5.1; "From sliding window to attention-guided
// eviction" §5.1): optionally update every token score with this step's
// attention -- exponential decay (score <- decay * score + increment), max
// over steps, or the exact sum over a sliding window of steps --, fold the
// tokens of each block into one block score (max, mean, the mean of the
// ceil(p * n) largest of the block's n valid tokens, the fraction of its
// tokens at or above a hotness threshold, or the max with only all-cold
// blocks evictable),
// normalise per request (the block's percentile inside its own request,
// fp32(2r + 1) / fp32(2n) for rank r by (score asc, block asc), or no
// normalisation), and emit the global eviction order: every block of every
// request sorted by (normalised score asc, request asc, block asc), the first
// ceil(frac * N) of them, as (request << 32) | block.
//
// Kernels (one call, four launches on the caller's stream):
//   bp_prefix_kernel  one CTA: blocks per request -> block offsets, N, the
//                     evict count; checks every length against the limits.
//   bp_fold_kernel    one warp per block (grid-stride): decay update of the
//                     block's tokens (written back) and the fold.
//   bp_rank_kernel    one CTA per request (percentile only): stable radix sort
//                     of the request's scores with block indices (up to 8192
//                     blocks; a register bitonic sort up to 16384; above that
//                     the same radix sort through global memory, 8192 keys a
//                     tile); the rank gives the percentile key of each block.
//   bp_sort_kernel    cooperative: stable LSD radix sort of the N 32-bit keys
//                     (4-bit digits, 8 passes, two bounded grid barriers per
//                     pass; the 16 digit offsets of a CTA are scanned at once).  The input is in (request, block) order and the
//                     sort is stable, so equal keys keep (request, block)
//                     order, which is the specified tie-break.  The first
//                     ceil(frac * N) codes go to the output.
#include "common.cuh"

namespace kvsel {

constexpr int kBpMaxBlockSize = 256;          // tokens per block: the pages' 16..256
constexpr int kBpMaxReqBlocks = 1 << 30;      // blocks per request: a block index fits the order code
constexpr int kBpSharedRankMax = 16384;       // blocks per request ranked in shared memory
constexpr int kBpSortThreads = 256;
constexpr int kBpMaxSortCtas = 256;

struct BpParams {
  float* tok;                // token scores (CSR by request), updated in place
  const float* inc;          // increments or null
  const int64_t* off;        // [R+1] token offsets
  float* bscore_out;         // [max_blocks] or null
  int64_t* order_out;        // [order_cap]
  int64_t* n_out;            // [2]: evict count, total blocks
  int64_t* blk_off;          // workspace [R+1]
  float* bscore;             // workspace [max_blocks]
  uint32_t* key[2];          // workspace [max_blocks] x 2
  int64_t* val[2];           // workspace [max_blocks] x 2
  int64_t* meta;             // workspace [3]: N (or -1), evict count, evictable (all-cold) blocks
  unsigned* hist;            // workspace [2][kBpMaxSortCtas][16]
  unsigned* bar;             // grid-barrier words
  int* status;
  int64_t max_blocks, order_cap;
  float* whist;              // WINDOW update: [window][hist_tokens] past increments
  long long step, hist_tokens;
  int R, bs, agg, norm, update, window;
  float decay, top_p, frac, threshold;
};

// aggregations (kvsel_block_agg; 2 = top-p mean) and updates (kvsel_score_update; 0 = decay)
constexpr int kAggMax = 0, kAggMean = 1, kAggFracHot = 3, kAggAllCold = 4;
constexpr int kUpdMax = 1, kUpdWindow = 2;

__device__ __forceinline__ int bp_request_of(const int64_t* blk_off, int R, int64_t g) {
  int lo = 0, hi = R - 1;  // last r with blk_off[r] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (blk_off[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(1024) bp_prefix_kernel(const BpParams P) {
  __shared__ long long warp_tot[33];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad = 0;
  __syncthreads();
  long long carry = 0;
  for (int base = 0; base < P.R; base += 1024) {
    const int r = base + tid;
    long long nb = 0;
    if (r < P.R) {
      const long long len = P.off[r + 1] - P.off[r];
      if (len < 0) bad = KVSEL_ERR_BAD_INDEX;
      nb = len > 0 ? (len + P.bs - 1) / P.bs : 0;
      if (nb > kBpMaxReqBlocks) bad = KVSEL_ERR_UNSUPPORTED;
    }
    long long x = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const long long t = warp_tot[lane];
      long long sc = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, sc, o);
        if (lane >= o) sc += y;
      }
      warp_tot[lane] = sc - t;
      if (lane == 31) warp_tot[32] = sc;
    }
    __syncthreads();
    if (r < P.R) P.blk_off[r] = carry + warp_tot[warp] + x - nb;
    carry += warp_tot[32];
    __syncthreads();
  }
  if (tid == 0) {
    P.blk_off[P.R] = carry;
    if (!bad && carry > P.max_blocks) bad = KVSEL_ERR_BAD_INDEX;
    if (!bad && P.inc && P.update == kUpdWindow && P.off[P.R] > P.hist_tokens) bad = KVSEL_ERR_BAD_INDEX;
    P.meta[2] = 0;
    const long long n_evict = bad ? 0 : (long long)ceil((double)P.frac * (double)carry);
    if (bad) report(P.status, bad);
    P.meta[0] = bad ? -1 : carry;
    P.meta[1] = n_evict;
    P.n_out[0] = n_evict;
    P.n_out[1] = bad ? -1 : carry;
  }
}

// One token's score update (decay, max over steps or the sliding-window sum), written back.
__device__ __forceinline__ float bp_update_token(const BpParams& P, float* hslot, long long t) {
  float s = P.tok[t];
  if (P.inc) {
    const float in = P.inc[t];
    if (P.update == kUpdMax) {
      s = fmaxf(s, in);
    } else if (P.update == kUpdWindow) {  // the increment leaving the window is replaced
      float* h = hslot + t;
      s = s + (in - *h);
      *h = in;
    } else {
      s = fmaf(P.decay, s, in);
    }
    P.tok[t] = s;
  }
  return s;
}

// The block's outputs (lane-independent): score, its copy out, the all-cold count, the sort key.
__device__ __forceinline__ void bp_block_out(const BpParams& P, long long g, int r, float result) {
  P.bscore[g] = result;
  if (P.bscore_out) P.bscore_out[g] = result;
  const bool hot_block = P.agg == kAggAllCold && result >= P.threshold;  // never evicted
  if (P.agg == kAggAllCold && !hot_block) atomicAdd(reinterpret_cast<unsigned long long*>(P.meta + 2), 1ull);
  if (P.norm == 0) {  // no normalisation: sort directly on the block score
    P.key[0][g] = hot_block ? 0xFFFFFFFFu : order_key(result);
    P.val[0][g] = ((long long)r << 32) | (g - P.blk_off[r]);
  }
}

// Blocks of up to 32 tokens: one lane per block.  A warp takes 32 consecutive blocks, whose tokens
// are one contiguous run of the CSR array (requests lie back to back): the warp loads, updates and
// writes that run back coalesced through its shared-memory buffer, then each lane folds its own
// block from there (a warp per block would have at most one block's 64..128 bytes in flight).
// The mean sums the block's scores in the lane's (rotated) visiting order, the top-p mean takes the
// maximum k times.
constexpr int kBpFoldThreads = 256;
__device__ __forceinline__ void bp_fold_lanes(const BpParams& P, long long N, float* hslot) {
  __shared__ float sbuf[kBpFoldThreads / 32][32 * 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* buf = sbuf[warp];
  const long long wstride = (long long)gridDim.x * (blockDim.x >> 5) * 32;
  for (long long g0 = ((long long)blockIdx.x * (blockDim.x >> 5) + warp) * 32; g0 < N; g0 += wstride) {
    const long long g = g0 + lane;
    const bool live = g < N;
    int r = 0, n = 0;
    long long t0 = 0;
    if (live) {
      r = bp_request_of(P.blk_off, P.R, g);
      t0 = P.off[r] + (g - P.blk_off[r]) * P.bs;
      n = int(min((long long)P.bs, P.off[r + 1] - t0));
    }
    const unsigned act = __ballot_sync(0xffffffffu, live);
    const int last = 31 - __clz(act);
    const long long T0 = __shfl_sync(0xffffffffu, t0, 0);
    const long long T1 = __shfl_sync(0xffffffffu, t0 + n, last);
    for (long long x = lane; x < T1 - T0; x += 32) buf[x] = bp_update_token(P, hslot, T0 + x);
    __syncwarp();
    float v[32];
    float sum = 0.f, mx = -INFINITY;
    int hot = 0;
    const int rel = int(t0 - T0);
    // each lane visits its block's tokens rotated by its lane index, so that lanes whose blocks
    // start a multiple of 32 words apart read different banks (the fold does not depend on order)
    const int rot = n > 0 ? lane % n : 0;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      v[t] = -INFINITY;
      if (t < n) {
        int q = t + rot;
        if (q >= n) q -= n;
        const float s = buf[rel + q];
        v[t] = s;
        sum += s;
        mx = fmaxf(mx, s);
        hot += s >= P.threshold ? 1 : 0;
      }
    }
    float result;
    if (P.agg == kAggMax || P.agg == kAggAllCold) {
      result = mx;
    } else if (P.agg == kAggFracHot) {
      result = __fdiv_rn(float(hot), float(n));
    } else if (P.agg == kAggMean) {
      result = __fdiv_rn(sum, float(n));
    } else {
      const int k = max(1, int(ceilf(__fmul_rn(P.top_p, float(n)))));
      float acc = 0.f;
      for (int it = 0; it < k; ++it) {  // the largest remaining, the lowest token on ties
        float m = -INFINITY;
        int at = 0;
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (v[t] > m) {
            m = v[t];
            at = t;
          }
        acc += m;
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t == at) v[t] = -INFINITY;
      }
      result = __fdiv_rn(acc, float(k));
    }
    if (live) bp_block_out(P, g, r, result);
    __syncwarp();  // every lane has read the buffer before the next group refills it
  }
}

__global__ void __launch_bounds__(kBpFoldThreads) bp_fold_kernel(const BpParams P) {
  const long long N = P.meta[0];
  if (N <= 0) return;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  constexpr int kPer = kBpMaxBlockSize / 32;
  // sliding-window update: this step's slot of the history ring
  float* const hslot = P.update == kUpdWindow ? P.whist + (P.step % P.window) * P.hist_tokens : nullptr;
  if (P.bs <= 32) {
    bp_fold_lanes(P, N, hslot);
    return;
  }
  for (long long g = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < N; g += warps) {
    const int r = bp_request_of(P.blk_off, P.R, g);
    const long long t0 = P.off[r] + (g - P.blk_off[r]) * P.bs;
    const int n = int(min((long long)P.bs, P.off[r + 1] - t0));
    float v[kPer];
    float sum = 0.f, mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int t = lane + 32 * e;
      v[e] = -INFINITY;
      if (t < n) {
        const float s = bp_update_token(P, hslot, t0 + t);
        v[e] = s;
        sum += s;
        mx = fmaxf(mx, s);
      }
    }
    float result;
    if (P.agg == kAggMax || P.agg == kAggAllCold) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      result = mx;
    } else if (P.agg == kAggFracHot) {  // fraction of valid tokens at or above the threshold
      int hot = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) hot += (lane + 32 * e < n && v[e] >= P.threshold) ? 1 : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) hot += __shfl_xor_sync(0xffffffffu, hot, o);
      result = __fdiv_rn(float(hot), float(n));
    } else if (P.agg == kAggMean) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      result = __fdiv_rn(sum, float(n));
    } else {
      // mean of the ceil(p * n) largest (p * n as an fp32 product): take the
      // warp maximum k times, removing one copy each time
      const int k = max(1, int(ceilf(__fmul_rn(P.top_p, float(n)))));
      float acc = 0.f;
      for (int it = 0; it < k; ++it) {
        float lm = -INFINITY;
        int le = 0;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
          if (v[e] > lm) {
            lm = v[e];
            le = e;
          }
        float wm = lm;
        int wl = lane;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, wm, o);
          const int ol = __shfl_xor_sync(0xffffffffu, wl, o);
          if (om > wm || (om == wm && ol < wl)) {
            wm = om;
            wl = ol;
          }
        }
        acc += wm;
        if (lane == wl) {
#pragma unroll
          for (int e = 0; e < kPer; ++e)
            if (e == le) v[e] = -INFINITY;
        }
      }
      result = __fdiv_rn(acc, float(k));
    }
    if (lane == 0) bp_block_out(P, g, r, result);
  }
}

// Bitonic sort of one request's (score key << 32 | block) keys, E per thread
// in registers (element i = thread * E + e): compare-exchanges inside a
// thread in registers, inside a warp through shuffles, and only those
// between warps through shared memory (one barrier pair each), then each
// block's percentile from its sorted position.
template <int E>
__device__ __forceinline__ void bp_rank_sort(unsigned long long* sk, int npow, int n, long long b0, int r,
                                             const BpParams& P) {
  const int tid = threadIdx.x;
  const bool act = tid * E < npow;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    v[e] = (act && i < n) ? ((unsigned long long)order_key(P.bscore[b0 + i]) << 32) | unsigned(i) : ~0ull;
  }
#pragma unroll 1
  for (int kk = 2; kk <= npow; kk <<= 1) {
#pragma unroll 1
    for (int jj = kk >> 1; jj >= E; jj >>= 1) {
      if (jj < 32 * E) {  // partner in another lane of this warp
        const int lx = jj / E;
        const bool lower = (tid & lx) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned long long p = __shfl_xor_sync(0xffffffffu, v[e], lx);
          const bool up = ((tid * E + e) & kk) == 0;
          v[e] = (up == lower) ? (v[e] < p ? v[e] : p) : (v[e] > p ? v[e] : p);
        }
      } else {  // partner in another warp
        __syncthreads();
        if (act) {
#pragma unroll
          for (int e = 0; e < E; ++e) sk[tid * E + e] = v[e];
        }
        __syncthreads();
        if (act) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int i = tid * E + e;
            const unsigned long long p = sk[i ^ jj];
            const bool up = (i & kk) == 0, lower = (i & jj) == 0;
            v[e] = (up == lower) ? (v[e] < p ? v[e] : p) : (v[e] > p ? v[e] : p);
          }
        }
      }
    }
    // partners in this thread: distances below E, unrolled so v stays in registers
#pragma unroll
    for (int jb = E / 2; jb >= 1; jb >>= 1) {
      if (jb < kk) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int l = e ^ jb;
          if (l > e) {
            const bool up = ((tid * E + e) & kk) == 0;
            const unsigned long long x = v[e], y = v[l];
            const bool sw = up ? (x > y) : (x < y);
            v[e] = sw ? y : x;
            v[l] = sw ? x : y;
          }
        }
      }
    }
  }
  if (act) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = tid * E + e;
      if (i < n) {
        const unsigned blk = unsigned(v[e] & 0xffffffffu);
        const float pct = __fdiv_rn(float(2 * i + 1), float(2 * n));  // correctly rounded
        const bool hot_block = P.agg == kAggAllCold && P.bscore[b0 + blk] >= P.threshold;
        P.key[0][b0 + blk] = hot_block ? 0xFFFFFFFFu : __float_as_uint(pct);  // pct > 0: bits are monotone
        P.val[0][b0 + blk] = ((long long)r << 32) | blk;
      }
    }
  }
}

// Stable LSD radix sort of one request's score keys (n <= 8192, 8-bit digits,
// 4 passes) with the block index as the value, then each block's percentile
// from its sorted position.  Thread t of warp w holds keys w*256 + e*32 + lane
// (e < 8), so a warp meets its keys in index order; per pass each warp ranks
// its keys among equal digits with match_any into a warp-private histogram
// column, one scan over (digit, warp) turns the columns into offsets, and the
// keys are scattered.  Equal scores keep block order, the specified tie-break.
constexpr int kRankRadixMax = 8192;
// A warp's histogram column is a row of 257 words: the leaders of one warp (different digits)
// then hit different banks, and the scan below, which walks (digit, warp) order 8 counts per
// thread, reads 32 distinct banks per instruction.
constexpr int kRankHistPitch = 257;
struct RankRadixSmem {
  uint32_t key[2][kRankRadixMax];
  uint16_t idx[2][kRankRadixMax];
  uint32_t hist[32 * kRankHistPitch];  // [warp][digit], padded: see kRankHistPitch
  uint32_t wsum[32];
};
__device__ __forceinline__ void bp_rank_radix(RankRadixSmem& sm, int n, long long b0, int r, const BpParams& P) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  uint32_t k[8];
  uint16_t v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int i = warp * 256 + e * 32 + lane;
    k[e] = i < n ? order_key(P.bscore[b0 + i]) : 0xFFFFFFFFu;  // padding sorts last
    v[e] = uint16_t(i);
  }
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    for (int j = tid; j < 32 * kRankHistPitch; j += 1024) sm.hist[j] = 0u;
    __syncthreads();
    uint32_t pos[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t d = (k[e] >> shift) & 255u;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      const int leader = __ffs(peers) - 1;
      uint32_t old = 0;
      if (lane == leader) {
        old = sm.hist[warp * kRankHistPitch + d];
        sm.hist[warp * kRankHistPitch + d] = old + __popc(peers);
      }
      pos[e] = __shfl_sync(0xffffffffu, old, leader) + __popc(peers & lt);
    }
    __syncthreads();
    {  // exclusive scan of the 8192 counts in (digit, warp) order: 8 per thread
      // count q = tid * 8 + j is digit q / 32 of warp q % 32
      auto at = [&](int q) -> uint32_t& { return sm.hist[(q & 31) * kRankHistPitch + (q >> 5)]; };
      uint32_t c[8], run = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = at(tid * 8 + j);
        run += c[j];
      }
      uint32_t incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) sm.wsum[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        const uint32_t t = sm.wsum[lane];
        uint32_t x = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        sm.wsum[lane] = x - t;
      }
      __syncthreads();
      uint32_t base = sm.wsum[warp] + incl - run;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        at(tid * 8 + j) = base;
        base += c[j];
      }
    }
    __syncthreads();
    const int ob = pass & 1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t d = (k[e] >> shift) & 255u;
      const uint32_t dst = sm.hist[warp * kRankHistPitch + d] + pos[e];
      sm.key[ob][dst] = k[e];
      sm.idx[ob][dst] = v[e];
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = warp * 256 + e * 32 + lane;
      k[e] = sm.key[ob][i];
      v[e] = sm.idx[ob][i];
    }
  }
  // after 4 passes position i holds the block of rank i (buffer 1)
  for (int i = tid; i < n; i += 1024) {
    const unsigned blk = sm.idx[1][i];
    const float pct = __fdiv_rn(float(2 * i + 1), float(2 * n));  // correctly rounded
    const bool hot_block = P.agg == kAggAllCold && P.bscore[b0 + blk] >= P.threshold;
    P.key[0][b0 + blk] = hot_block ? 0xFFFFFFFFu : __float_as_uint(pct);  // pct > 0: bits are monotone
    P.val[0][b0 + blk] = ((long long)r << 32) | blk;
  }
}

// Requests above kBpSharedRankMax blocks: the same stable LSD radix sort (8-bit digits, 4
// passes), its keys and block indices ping-ponging through the request's own segments of the
// workspace key / value arrays (the global sort only uses them afterwards).  A pass first counts
// every digit over the request, then visits the request in tiles of 8192 keys in order; inside a
// tile the keys are ranked among equal digits exactly as in bp_rank_radix, and a key goes to its
// digit's next free slot plus its rank among that digit's keys in the tile.  Tiles in order and
// ranks in index order keep the sort stable.
struct RankGlobalSmem {
  uint32_t hist[32 * kRankHistPitch];  // [warp][digit], padded; slot 256 takes the tail's empty lanes
  uint32_t wsum[32];
  uint32_t run[256];                   // the next output slot of each digit
  uint32_t tstart[257];                // the tile's first slot of each digit; [256]: its keys
};
__device__ __forceinline__ void bp_rank_global(RankGlobalSmem& sm, int n, long long b0, int r, const BpParams& P) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  uint32_t* kb[2] = {P.key[0] + b0, P.key[1] + b0};
  int64_t* vb[2] = {P.val[0] + b0, P.val[1] + b0};
  const int tiles = (n + kRankRadixMax - 1) / kRankRadixMax;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    const int dstb = (pass & 1) ^ 1, srcb = pass & 1;  // pass 0 reads the scores: 1, 0, 1, 0
    auto key_at = [&](int i) -> uint32_t { return pass == 0 ? order_key(P.bscore[b0 + i]) : kb[srcb][i]; };
    auto val_at = [&](int i) -> uint32_t { return pass == 0 ? uint32_t(i) : uint32_t(vb[srcb][i]); };
    // every digit's count over the request, then each digit's first slot
    if (tid < 256) sm.run[tid] = 0u;
    __syncthreads();
    for (int i0 = warp * 32; i0 < n; i0 += 1024) {  // lanes with the same digit add once
      const int i = i0 + lane;
      const uint32_t d = i < n ? (key_at(i) >> shift) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (d < 256u && lane == __ffs(peers) - 1) atomicAdd(&sm.run[d], uint32_t(__popc(peers)));
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.run[lane * 8 + j];
        tot += c[j];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t base = incl - tot;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sm.run[lane * 8 + j] = base;
        base += c[j];
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int t = 0; t < tiles; ++t) {
      const int t0 = t * kRankRadixMax;
      for (int j = tid; j < 32 * kRankHistPitch; j += 1024) sm.hist[j] = 0u;
      __syncthreads();
      uint32_t k[8], v[8], pos[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = t0 + warp * 256 + e * 32 + lane;
        const bool ok = i < n;
        k[e] = ok ? key_at(i) : 0u;
        v[e] = ok ? val_at(i) : 0u;
        const uint32_t d = ok ? (k[e] >> shift) & 255u : 256u;  // past the end: the unused slot 256
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const int leader = __ffs(peers) - 1;
        uint32_t old = 0;
        if (lane == leader) {
          old = sm.hist[warp * kRankHistPitch + d];
          sm.hist[warp * kRankHistPitch + d] = old + __popc(peers);
        }
        pos[e] = __shfl_sync(0xffffffffu, old, leader) + __popc(peers & lt);
      }
      __syncthreads();
      {  // exclusive scan of the tile's 8192 counts in (digit, warp) order: 8 per thread
        auto at = [&](int q) -> uint32_t& { return sm.hist[(q & 31) * kRankHistPitch + (q >> 5)]; };
        uint32_t c[8], run = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = at(tid * 8 + j);
          run += c[j];
        }
        uint32_t incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) sm.wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
          const uint32_t tw = sm.wsum[lane];
          uint32_t x = tw;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          sm.wsum[lane] = x - tw;
        }
        __syncthreads();
        uint32_t base = sm.wsum[warp] + incl - run;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          at(tid * 8 + j) = base;
          base += c[j];
        }
      }
      __syncthreads();
      if (tid < 256) sm.tstart[tid] = sm.hist[tid];  // warp 0's column: where digit tid starts in the tile
      if (tid == 0) sm.tstart[256] = uint32_t(min(kRankRadixMax, n - t0));
      __syncthreads();
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = t0 + warp * 256 + e * 32 + lane;
        if (i < n) {
          const uint32_t d = (k[e] >> shift) & 255u;
          const uint32_t dst = sm.run[d] + sm.hist[warp * kRankHistPitch + d] + pos[e] - sm.tstart[d];
          kb[dstb][dst] = k[e];
          vb[dstb][dst] = v[e];
        }
      }
      __syncthreads();
      if (tid < 256) sm.run[tid] += sm.tstart[tid + 1] - sm.tstart[tid];  // the digit's keys in this tile
      __syncthreads();
    }
  }
  // buffer 0 holds the blocks in rank order: their indices move to key buffer 1 before buffer 0
  // is overwritten with the percentile keys
  for (int i = tid; i < n; i += 1024) kb[1][i] = uint32_t(vb[0][i]);
  __syncthreads();
  for (int i = tid; i < n; i += 1024) {
    const unsigned blk = kb[1][i];
    const float pct = __fdiv_rn(__ll2float_rn(2LL * i + 1), __ll2float_rn(2LL * n));  // correctly rounded
    const bool hot_block = P.agg == kAggAllCold && P.bscore[b0 + blk] >= P.threshold;
    P.key[0][b0 + blk] = hot_block ? 0xFFFFFFFFu : __float_as_uint(pct);
    P.val[0][b0 + blk] = ((long long)r << 32) | blk;
  }
}

__global__ void __launch_bounds__(1024) bp_rank_kernel(const BpParams P) {
  extern __shared__ unsigned long long skeys[];
  if (P.meta[0] <= 0) return;
  const int r = blockIdx.x;
  const long long b0 = P.blk_off[r];
  const int n = int(P.blk_off[r + 1] - b0);
  if (n == 0) return;
  if (n <= kRankRadixMax) {
    bp_rank_radix(*reinterpret_cast<RankRadixSmem*>(skeys), n, b0, r, P);
    return;
  }
  if (n > kBpSharedRankMax) {
    bp_rank_global(*reinterpret_cast<RankGlobalSmem*>(skeys), n, b0, r, P);
    return;
  }
  int npow = 1;
  while (npow < n) npow <<= 1;
  switch (npow <= 1024 ? 1 : npow / 1024) {  // keys per thread (bitonic, requests above 8192 blocks)
    case 1: bp_rank_sort<1>(skeys, npow, n, b0, r, P); break;
    case 2: bp_rank_sort<2>(skeys, npow, n, b0, r, P); break;
    case 4: bp_rank_sort<4>(skeys, npow, n, b0, r, P); break;
    case 8: bp_rank_sort<8>(skeys, npow, n, b0, r, P); break;
    default: bp_rank_sort<16>(skeys, npow, n, b0, r, P); break;
  }
}

// Grid barrier of the cooperative sort: 2^26 sleeps of ~32 ns (a few
// seconds) unless the workspace sets another limit.  Returns false, in every
// thread of the CTA, when the wait ran out (KVSEL_ERR_TIMEOUT recorded): the
// caller must then stop, since the digit offsets it would scatter with may
// be incomplete.
__device__ __forceinline__ bool bp_grid_barrier(unsigned* bar, int* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile unsigned* gen = bar + 32;
    const unsigned g = *gen;
    __threadfence();
    if (atomicAdd(bar, 1u) + 1u == gridDim.x) {
      bar[0] = 0u;
      __threadfence();
      atomicAdd(bar + 32, 1u);
    } else {
      const unsigned limit = spin_limit(status, 1u << 26);
      unsigned spins = 0;
      while (*gen == g) {
        __nanosleep(32);
        if (++spins >= limit) {
          report(status, KVSEL_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__global__ void __launch_bounds__(kBpSortThreads) bp_sort_kernel(const BpParams P) {
  __shared__ unsigned cnt[16][kBpSortThreads];
  __shared__ unsigned base[16];
  __shared__ unsigned sTot[kBpSortThreads / 16][16], sBefore[kBpSortThreads / 16][16];
  __shared__ unsigned wtot[kBpSortThreads / 32][16];
  __shared__ int s_same;
  const long long N = P.meta[0];
  if (N < 0) return;  // same for every CTA
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = gridDim.x, c = blockIdx.x;
  const long long c0 = N * c / NC, c1 = N * (c + 1) / NC;
  const long long per = (c1 - c0 + kBpSortThreads - 1) / kBpSortThreads;
  const long long t0 = min(c1, c0 + per * tid), t1 = min(c1, t0 + per);

  int cur = 0;  // the buffer holding the keys sorted so far
#pragma unroll 1
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 4 * pass;
    const uint32_t* ik = P.key[cur];
    const int64_t* iv = P.val[cur];
    uint32_t* ok = P.key[cur ^ 1];
    int64_t* ov = P.val[cur ^ 1];
    // the CTAs' digit counts alternate between two halves: a pass whose scatter is skipped has no
    // second barrier, so a CTA may write the next pass's counts while another still reads these
    unsigned* phist = P.hist + (pass & 1) * (kBpMaxSortCtas * 16);
    // this thread's digit counts (its keys are a contiguous run of the input)
    unsigned v[16];
#pragma unroll
    for (int d = 0; d < 16; ++d) v[d] = 0u;
    for (long long e = t0; e < t1; ++e) {
      const unsigned dd = (ik[e] >> shift) & 15u;
#pragma unroll
      for (int d = 0; d < 16; ++d) v[d] += dd == unsigned(d) ? 1u : 0u;
    }
    // all 16 digits scanned at once: inclusive over the warp's lanes, then the
    // 8 warp totals of each digit by one thread per digit
    unsigned x[16];
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      x[d] = v[d];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x[d], o);
        if (lane >= o) x[d] += y;
      }
    }
    if (lane == 31) {
#pragma unroll
      for (int d = 0; d < 16; ++d) wtot[warp][d] = x[d];
    }
    __syncthreads();
    if (tid < 16) {
      unsigned run = 0;
      for (int w = 0; w < kBpSortThreads / 32; ++w) {
        const unsigned t = wtot[w][tid];
        wtot[w][tid] = run;
        run += t;
      }
      phist[c * 16 + tid] = run;  // this CTA's count of digit tid
    }
    __syncthreads();
#pragma unroll
    for (int d = 0; d < 16; ++d) cnt[d][tid] = wtot[warp][d] + x[d] - v[d];  // exclusive offset inside this CTA
    if (!bp_grid_barrier(P.bar, P.status)) return;  // timed out: stop before any scatter
    {
      // start of digit d for this CTA = all keys with a smaller digit + this
      // digit's keys in earlier CTAs; 16 stripes of CTAs x 16 digits in parallel
      const int d = tid & 15, stripe = tid >> 4;
      unsigned tot = 0, before = 0;
      for (int cc = stripe; cc < NC; cc += kBpSortThreads / 16) {
        const unsigned h = __ldcg(phist + cc * 16 + d);
        tot += h;
        if (cc < c) before += h;
      }
      sTot[stripe][d] = tot;
      sBefore[stripe][d] = before;
      __syncthreads();
      if (tid < 16) {
        unsigned t = 0, b = 0;
        for (int st = 0; st < kBpSortThreads / 16; ++st) {
          t += sTot[st][tid];
          b += sBefore[st][tid];
        }
        sTot[0][tid] = t;   // digit totals (read below by thread 0 only after the sync)
        base[tid] = b;
      }
      __syncthreads();
      if (tid == 0) {
        unsigned run = 0, widest = 0;
        for (int dd = 0; dd < 16; ++dd) {
          const unsigned t = sTot[0][dd];
          base[dd] += run;
          run += t;
          widest = max(widest, t);
        }
        s_same = widest == run;  // one digit holds every key: the stable scatter would not move one
      }
    }
    __syncthreads();
    if (s_same) continue;  // the same in every CTA: no scatter, no barrier, the keys stay where they are
    for (long long e = t0; e < t1; ++e) {
      const uint32_t k = ik[e];
      const unsigned d = (k >> shift) & 15u;
      const unsigned pos = base[d] + cnt[d][tid]++;
      ok[pos] = k;
      ov[pos] = iv[e];
    }
    if (!bp_grid_barrier(P.bar, P.status)) return;  // timed out: stop before any scatter
    cur ^= 1;
  }
  long long n_all = P.meta[1];
  if (P.agg == kAggAllCold) {  // only the evictable blocks (they sort first)
    n_all = min(n_all, (long long)P.meta[2]);
    if (c == 0 && tid == 0) P.n_out[0] = n_all;
  }
  const long long n_ev = min(n_all, (long long)P.order_cap);
  for (long long i = (long long)c * kBpSortThreads + tid; i < n_ev; i += (long long)NC * kBpSortThreads)
    P.order_out[i] = __ldcg(P.val[cur] + i);
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct BpWs {
  size_t blk_off, bscore, key0, key1, val0, val1, meta, hist, total;
};
BpWs bp_ws_layout(int R, long long max_blocks) {
  BpWs w;
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.blk_off = take(size_t(R + 1) * 8);
  w.bscore = take(size_t(max_blocks) * 4);
  w.key0 = take(size_t(max_blocks) * 4);
  w.key1 = take(size_t(max_blocks) * 4);
  w.val0 = take(size_t(max_blocks) * 8);
  w.val1 = take(size_t(max_blocks) * 8);
  w.meta = take(24);
  w.hist = take(size_t(2) * kBpMaxSortCtas * 16 * 4);
  w.total = off;
  return w;
}
}  // namespace

extern "C" size_t kvsel_block_priority_workspace(int num_requests, int64_t max_total_blocks) {
  if (num_requests < 1 || max_total_blocks < 1) return 0;
  return bp_ws_layout(num_requests, max_total_blocks).total;
}

extern "C" kvsel_status kvsel_block_priority(float* token_scores, const float* increment, float decay,
                                             const int64_t* req_offsets, int num_requests, int block_size,
                                             int agg, float top_p, int norm, float evict_frac,
                                             float* block_score_out, int64_t max_total_blocks,
                                             int64_t* order_out, int64_t order_capacity, int64_t* n_out,
                                             void* workspace, size_t ws_bytes, void* stream) {
  if (agg == KVSEL_AGG_FRAC_HOT || agg == KVSEL_AGG_ALL_COLD)
    return fail(KVSEL_ERR_INVALID_ARG, "kvsel_block_priority: the threshold aggregations need kvsel_block_priority_ex");
  return kvsel_block_priority_ex(token_scores, increment, decay, req_offsets, num_requests, block_size, agg, top_p,
                                 norm, evict_frac, block_score_out, max_total_blocks, order_out, order_capacity,
                                 n_out, workspace, ws_bytes, nullptr, stream);
}

extern "C" kvsel_status kvsel_block_priority_ex(float* token_scores, const float* increment, float decay,
                                                const int64_t* req_offsets, int num_requests, int block_size,
                                                int agg, float top_p, int norm, float evict_frac,
                                                float* block_score_out, int64_t max_total_blocks,
                                                int64_t* order_out, int64_t order_capacity, int64_t* n_out,
                                                void* workspace, size_t ws_bytes, const kvsel_bp_options* opt,
                                                void* stream) {
  const std::string fn = "kvsel_block_priority: ";
  kvsel_bp_options o = {};
  o.update = KVSEL_UPDATE_DECAY;
  if (opt) o = *opt;
  if (o.update < KVSEL_UPDATE_DECAY || o.update > KVSEL_UPDATE_WINDOW)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "update must be KVSEL_UPDATE_DECAY, _MAX or _WINDOW");
  if (increment && o.update == KVSEL_UPDATE_WINDOW &&
      (!o.history || o.window < 1 || o.step < 0 || o.history_tokens < 1 || !aligned(o.history, 4)))
    return fail(KVSEL_ERR_INVALID_ARG,
                fn + "the window update needs history, window >= 1, step >= 0 and history_tokens >= 1");
  if ((agg == KVSEL_AGG_FRAC_HOT || agg == KVSEL_AGG_ALL_COLD) && !(o.threshold == o.threshold))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "threshold must be a number");
  if (!token_scores || !req_offsets || !n_out || num_requests < 1 || max_total_blocks < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "token_scores, req_offsets, n_out are required; num_requests, "
                                            "max_total_blocks >= 1");
  if (block_size < 1 || block_size > kBpMaxBlockSize)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "block_size must be in [1, 256]");
  if (agg < KVSEL_AGG_MAX || agg > KVSEL_AGG_ALL_COLD)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "agg must be KVSEL_AGG_MAX, _MEAN, _TOPP, _FRAC_HOT or _ALL_COLD");
  if (norm != KVSEL_NORM_NONE && norm != KVSEL_NORM_PERCENTILE)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "norm must be KVSEL_NORM_NONE or KVSEL_NORM_PERCENTILE");
  if (agg == KVSEL_AGG_TOPP && !(top_p > 0.f && top_p <= 1.f))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "top_p must be in (0, 1]");
  if (!(evict_frac >= 0.f && evict_frac <= 1.f))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "evict_frac must be in [0, 1]");
  if (increment && o.update == KVSEL_UPDATE_DECAY && !(decay == decay))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "decay must be a number");
  if (order_capacity < 0 || (order_capacity > 0 && !order_out))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "order_out is required when order_capacity > 0");
  if (max_total_blocks >= (1LL << 31))
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 2^31 - 1 blocks");
  if (!workspace || !aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "a 256-byte aligned workspace is required");
  const BpWs L = bp_ws_layout(num_requests, max_total_blocks);
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(L.total));

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BpParams P;
  P.tok = token_scores;
  P.inc = increment;
  P.off = req_offsets;
  P.bscore_out = block_score_out;
  P.order_out = order_out;
  P.n_out = n_out;
  P.blk_off = reinterpret_cast<int64_t*>(ws + L.blk_off);
  P.bscore = reinterpret_cast<float*>(ws + L.bscore);
  P.key[0] = reinterpret_cast<uint32_t*>(ws + L.key0);
  P.key[1] = reinterpret_cast<uint32_t*>(ws + L.key1);
  P.val[0] = reinterpret_cast<int64_t*>(ws + L.val0);
  P.val[1] = reinterpret_cast<int64_t*>(ws + L.val1);
  P.meta = reinterpret_cast<int64_t*>(ws + L.meta);
  P.hist = reinterpret_cast<unsigned*>(ws + L.hist);
  P.bar = reinterpret_cast<unsigned*>(ws + 64);
  P.status = reinterpret_cast<int*>(ws);
  P.max_blocks = max_total_blocks;
  P.order_cap = order_capacity;
  P.R = num_requests;
  P.bs = block_size;
  P.agg = agg;
  P.norm = norm;
  P.decay = decay;
  P.top_p = top_p;
  P.frac = evict_frac;
  P.update = o.update;
  P.whist = o.history;
  P.window = o.window > 0 ? o.window : 1;
  P.step = o.step;
  P.hist_tokens = o.history_tokens;
  P.threshold = o.threshold;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  trace_before("bp_prefix", st);
  bp_prefix_kernel<<<1, 1024, 0, st>>>(P);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_block_priority (prefix launch)");

  const int sms = sm_count();
  trace_before("bp_fold", st);
  bp_fold_kernel<<<sms * 8, kBpFoldThreads, 0, st>>>(P);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_block_priority (fold launch)");

  if (norm == KVSEL_NORM_PERCENTILE) {
    const size_t smem =
        std::max(std::max(size_t(kBpSharedRankMax) * 8, sizeof(RankRadixSmem)), sizeof(RankGlobalSmem));
    static bool attr_set = false;
    if (!attr_set) {
      e = cudaFuncSetAttribute(bp_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return cuda_fail(e, "kvsel_block_priority (rank attribute)");
      attr_set = true;
    }
    trace_before("bp_rank", st);
    bp_rank_kernel<<<num_requests, 1024, smem, st>>>(P);
    e = cudaGetLastError();
    trace_after(st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_block_priority (rank launch)");
  }

  // cooperative sort: CTAs co-resident (<= one per SM here), ~2K keys per CTA
  int nc = int(std::min<long long>((max_total_blocks + 2047) / 2048, (long long)sms));
  nc = std::max(1, std::min(nc, kBpMaxSortCtas));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc);
  cfg.blockDim = dim3(kBpSortThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before("bp_sort", st);
  e = cudaLaunchKernelEx(&cfg, bp_sort_kernel, P);
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_block_priority (sort launch)");
  return KVSEL_OK;
}
