// Exact block-wide top-k over keys held in registers (sm_103a).
//
// Each thread of a 1024-thread CTA holds a contiguous run of at most kItems
// candidates (monotone uint32 keys, larger = better), runs laid out in
// position order.  block_topk_threshold finds the k-th largest key T and how
// many keys equal to T belong to the top k (the lowest positions win ties):
// a sorted sample (the first key of every run) brackets T between two sample
// quantiles with a margin of four binomial standard deviations, one counting
// pass checks the bracket, the keys inside it are gathered to shared memory
// and a 4 x 8-bit radix select finishes exactly.  If the bracket misses, a
// radix select over all the register runs runs instead.  The caller then
// emits the kept items in position order with block_topk_emit_offsets.
#pragma once

#include "common.cuh"

namespace kvsel {

constexpr int kTopkThreads = 1024;
constexpr int kTopkBandMax = 8192;

struct TopkCore {
  uint32_t hist[256];
  uint32_t scan[33];
  uint32_t digit, above;
  uint32_t sample[kTopkThreads];
};
struct TopkSmem : TopkCore {
  uint32_t band[kTopkBandMax];
};

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ __forceinline__ uint32_t topk_block_scan(uint32_t v, uint32_t* tmp, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = tmp[lane];
    uint32_t s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    tmp[lane] = s - t;
    if (lane == 31) tmp[32] = s;
  }
  __syncthreads();
  const uint32_t r = tmp[warp] + x - v;
  total = tmp[32];
  __syncthreads();
  return r;
}

// One radix-select digit decision: warp 0 scans the 256-bin histogram from the
// top and records the digit holding the krem-th largest and the count above it.
__device__ __forceinline__ void topk_pick_digit(TopkCore& sm, uint32_t krem) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) == 0) {
    uint32_t cb[8], lsum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cb[e] = sm.hist[255 - 8 * lane - e];
      lsum += cb[e];
    }
    uint32_t incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - lsum;
    if (excl < krem && krem <= incl) {
      uint32_t above = excl;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (above + cb[e] >= krem) {
          sm.digit = 255 - 8 * lane - e;
          sm.above = above;
          break;
        }
        above += cb[e];
      }
    }
  }
}

// k-th largest of all threads' valid keys (key[e] for e < cnt); 1 <= k <= total.
template <int kItems>
__device__ __forceinline__ void block_topk_threshold(const uint32_t (&key)[kItems], int cnt,
                                                     int n_total, int k, TopkSmem& sm, uint32_t& T,
                                                     uint32_t& need_eq) {
  const int tid = threadIdx.x;
  // 1. sorted sample: first key of every run (0 sorts below every real key)
  sm.sample[tid] = cnt > 0 ? key[0] : 0u;
  __syncthreads();
  for (int kk = 2; kk <= kTopkThreads; kk <<= 1)
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      const int l = tid ^ jj;
      if (l > tid) {
        const uint32_t x = sm.sample[tid], y = sm.sample[l];
        const bool desc = (tid & kk) == 0;
        if (desc ? (x < y) : (x > y)) {
          sm.sample[tid] = y;
          sm.sample[l] = x;
        }
      }
      __syncthreads();
    }
  // 2. bracket around the estimated sample rank of the k-th key
  const int C = (n_total + kTopkThreads - 1) / kTopkThreads;
  const int ns = (n_total + C - 1) / C;
  const float p = float(k) / float(n_total);
  const int est = int((long long)k * ns / n_total);
  const int margin = 16 + int(4.0f * sqrtf(float(ns) * p * (1.f - p)));
  const uint32_t t_hi = est - margin >= 0 ? sm.sample[est - margin] : 0xFFFFFFFFu;
  const uint32_t t_lo = est + margin < ns ? sm.sample[est + margin] : 0u;
  uint32_t c_gt = 0, c_band = 0;
#pragma unroll
  for (int e = 0; e < kItems; ++e)
    if (e < cnt) {
      c_gt += key[e] > t_hi;
      c_band += (key[e] >= t_lo) & (key[e] <= t_hi);
    }
  uint32_t gt_tot, band_tot;
  topk_block_scan(c_gt, sm.scan, gt_tot);
  const uint32_t band_base = topk_block_scan(c_band, sm.scan, band_tot);
  const bool bracket_ok =
      gt_tot < uint32_t(k) && uint32_t(k) <= gt_tot + band_tot && band_tot <= uint32_t(kTopkBandMax);
  uint32_t krem = bracket_ok ? uint32_t(k) - gt_tot : uint32_t(k);
  if (bracket_ok) {
    uint32_t w = band_base;
#pragma unroll
    for (int e = 0; e < kItems; ++e)
      if (e < cnt && (key[e] >= t_lo) & (key[e] <= t_hi)) sm.band[w++] = key[e];
  }
  __syncthreads();
  // 3. radix select over the band (or, if the bracket missed, over every key)
  uint32_t prefix = 0, mask = 0;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) sm.hist[tid] = 0;
    __syncthreads();
    if (bracket_ok) {
      for (uint32_t i = tid; i < band_tot; i += kTopkThreads) {
        const uint32_t u = sm.band[i];
        if ((u & mask) == prefix) atomicAdd(&sm.hist[(u >> shift) & 255u], 1u);
      }
    } else {
#pragma unroll
      for (int e = 0; e < kItems; ++e)
        if (e < cnt && (key[e] & mask) == prefix) atomicAdd(&sm.hist[(key[e] >> shift) & 255u], 1u);
    }
    __syncthreads();
    topk_pick_digit(sm, krem);
    __syncthreads();
    krem -= sm.above;
    prefix |= sm.digit << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  T = prefix;
  need_eq = krem;
}

// Given (T, need_eq): this thread's number of kept items and its output offset
// (items are kept in position order: keys > T, and the first need_eq keys == T).
template <int kItems>
__device__ __forceinline__ uint32_t block_topk_emit_offsets(const uint32_t (&key)[kItems], int cnt,
                                                           uint32_t T, uint32_t need_eq,
                                                           TopkSmem& sm, uint32_t& eq_rank0) {
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int e = 0; e < kItems; ++e)
    if (e < cnt) {
      gt += key[e] > T;
      eq += key[e] == T;
    }
  uint32_t tot;
  eq_rank0 = topk_block_scan(eq, sm.scan, tot);
  const uint32_t take_eq = need_eq > eq_rank0 ? min(eq, need_eq - eq_rank0) : 0u;
  return topk_block_scan(gt + take_eq, sm.scan, tot);
}

}  // namespace kvsel

namespace kvsel {

// ---------------------------------------------------------------------------
// Top-k positions through the "upper set".
//
// A lower bound t_lo on the k-th key (a caller hint, else a sample quantile
// k/n + four binomial standard deviations below the estimate) selects the
// keys >= t_lo; one counting pass and one gather move them, with their
// positions and in position order, into shared memory.  When that set holds
// at least k and at most kUpMax keys, the exact radix select and the ordered
// emission run over it alone.  Otherwise the caller falls back to the
// register-run path above.
// ---------------------------------------------------------------------------
constexpr int kUpMax = 12288;

struct UpperSmem {
  TopkCore base;            // histogram, scans, sample
  uint32_t ukey[kUpMax];
  int32_t upos[kUpMax];
};
// Dynamic shared memory big enough for either the register-run path (TopkSmem)
// or the upper-set path (UpperSmem); both views alias the same bytes.
constexpr size_t kTopkDynSmem = sizeof(UpperSmem) > sizeof(TopkSmem) ? sizeof(UpperSmem) : sizeof(TopkSmem);

// Returns true and writes the k kept positions (ascending) to out[0..k), with
// T / need_eq describing the threshold, or returns false (nothing written).
template <int kItems, class PosFn>
__device__ __forceinline__ bool block_topk_upper(const uint32_t (&key)[kItems], int cnt, PosFn pos_of,
                                                 int n_total, int k, uint32_t hint, UpperSmem& sm,
                                                 int32_t* out, uint32_t& T, uint32_t& need_eq) {
  const int tid = threadIdx.x;
  uint32_t t_lo = hint;
  if (t_lo == 0u) {
    // sample quantile below the estimated rank of the k-th key
    sm.base.sample[tid] = cnt > 0 ? key[0] : 0u;
    __syncthreads();
    for (int kk = 2; kk <= kTopkThreads; kk <<= 1)
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        const int l = tid ^ jj;
        if (l > tid) {
          const uint32_t x = sm.base.sample[tid], y = sm.base.sample[l];
          const bool desc = (tid & kk) == 0;
          if (desc ? (x < y) : (x > y)) {
            sm.base.sample[tid] = y;
            sm.base.sample[l] = x;
          }
        }
        __syncthreads();
      }
    const int C = (n_total + kTopkThreads - 1) / kTopkThreads;
    const int ns = (n_total + C - 1) / C;
    const float p = float(k) / float(n_total);
    const int est = int((long long)k * ns / n_total);
    const int margin = 16 + int(4.0f * sqrtf(float(ns) * p * (1.f - p)));
    t_lo = est + margin < ns ? sm.base.sample[est + margin] : 0u;
  }
  uint32_t c_up = 0;
#pragma unroll
  for (int e = 0; e < kItems; ++e)
    if (e < cnt) c_up += key[e] >= t_lo;
  uint32_t up_tot;
  const uint32_t base = topk_block_scan(c_up, sm.base.scan, up_tot);
  if (up_tot < uint32_t(k) || up_tot > uint32_t(kUpMax)) return false;  // uniform over the block
  {
    uint32_t w = base;
#pragma unroll
    for (int e = 0; e < kItems; ++e)
      if (e < cnt && key[e] >= t_lo) {
        sm.ukey[w] = key[e];
        sm.upos[w] = pos_of(e);
        ++w;
      }
  }
  __syncthreads();
  // exact k-th key inside the upper set
  uint32_t prefix = 0, mask = 0, krem = uint32_t(k);
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) sm.base.hist[tid] = 0;
    __syncthreads();
    for (uint32_t i = tid; i < up_tot; i += kTopkThreads) {
      const uint32_t u = sm.ukey[i];
      if ((u & mask) == prefix) atomicAdd(&sm.base.hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    topk_pick_digit(sm.base, krem);
    __syncthreads();
    krem -= sm.base.above;
    prefix |= sm.base.digit << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  T = prefix;
  need_eq = krem;
  // ordered emission over the upper set: contiguous runs per thread
  const int C = (int(up_tot) + kTopkThreads - 1) / kTopkThreads;
  const int i0 = min(int(up_tot), tid * C), i1 = min(int(up_tot), (tid + 1) * C);
  uint32_t gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    gt += sm.ukey[i] > T;
    eq += sm.ukey[i] == T;
  }
  uint32_t tot;
  const uint32_t eq_base = topk_block_scan(eq, sm.base.scan, tot);
  const uint32_t take_eq = need_eq > eq_base ? min(eq, need_eq - eq_base) : 0u;
  uint32_t w = topk_block_scan(gt + take_eq, sm.base.scan, tot);
  uint32_t q = eq_base;
  for (int i = i0; i < i1; ++i) {
    const uint32_t u = sm.ukey[i];
    const bool isq = u == T;
    if ((u > T || (isq && q < need_eq)) && w < uint32_t(k)) out[w++] = sm.upos[i];
    q += isq;
  }
  return true;
}

}  // namespace kvsel
