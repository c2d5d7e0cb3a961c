// Exact top-k of one row per 1024-thread CTA, kept positions emitted in
// ascending order (sm_103a).
//
// Keys are monotone uint32 images of the scores (larger = better); key 0
// marks "no candidate" (no finite float maps to it).  Ties at the k-th key go
// to the lower positions.
//
// Layout: the row's relative positions [0, n) are cut into 32 contiguous warp
// segments of L positions (L a multiple of 128); inside a segment a warp
// walks groups of 128 positions, lane l holding positions 4l .. 4l+3 of the
// group, so every load is one coalesced 512-byte float4 access.  Segments of
// up to kG groups stay in registers for the whole selection; longer ones are
// swept kG groups at a time and re-read (from L2) on each sweep.
//
// Steps:
//   1. a lower bound t_lo on the k-th key: the caller's hint (the previous
//      call's threshold) if it works, else a quantile of a 1024-key systematic
//      sample (found by the same radix select), four binomial standard
//      deviations below the estimated rank;
//   2. one sweep gathers the keys >= t_lo (the "upper set", order free) into
//      shared memory with one atomic reservation per warp, and their maximum;
//   3. radix select of the k-th key over the upper set, 8-bit digits starting
//      below the bits that t_lo and the maximum share; the histogram keeps a
//      private column per lane, so skewed digits never collide in a warp;
//   4. ordered emission: per-warp counts of keys > T and == T, one block
//      exchange of the 32 warp totals, then a ballot-ordered pass per group
//      that stages the kept positions in shared memory (k <= 16384), so the
//      caller's outputs are written with consecutive threads on consecutive
//      entries.
// When the upper set is too small (the bound was above the k-th key) or too
// large for shared memory, a radix select over the whole row replaces 2-3.
#pragma once

#include "common.cuh"

namespace kvsel {

constexpr int kRkThreads = 1024;
constexpr int kRkUpMax = 16384;  // upper-set capacity (keys)

struct RowTopkSmem {
  uint32_t lhist[256][32];  // radix histogram, one column per lane
  uint32_t hist[256];
  uint32_t wtot[2][32];
  uint32_t cnt, maxkey, digit, above;
  uint32_t ukey[kRkUpMax];
};

// Keys of an fp32 row p[0..n) (relative positions), valid for lo <= rel < n.
struct F32RowKeys {
  const float* p;
  int lo, n;
  bool vec;  // p is 16-byte aligned
  __device__ __forceinline__ uint32_t load1(int rel) const {
    return (rel >= lo && rel < n) ? order_key(__ldcg(p + rel)) : 0u;
  }
  __device__ __forceinline__ uint4 load4(int rel) const {
    uint4 k;
    if (vec && rel + 3 < n && rel >= lo) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p + rel));
      k = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
    } else {
      k = make_uint4(load1(rel), load1(rel + 1), load1(rel + 2), load1(rel + 3));
    }
    return k;
  }
};

// Precomputed keys q[0..n) (relative positions), valid for lo <= rel < n.
struct U32RowKeys {
  const uint32_t* q;
  int lo, n;
  bool vec;
  __device__ __forceinline__ uint32_t load1(int rel) const {
    return (rel >= lo && rel < n) ? __ldcg(q + rel) : 0u;
  }
  __device__ __forceinline__ uint4 load4(int rel) const {
    if (vec && rel + 3 < n && rel >= lo) return __ldcg(reinterpret_cast<const uint4*>(q + rel));
    return make_uint4(load1(rel), load1(rel + 1), load1(rel + 2), load1(rel + 3));
  }
};

// Positions per warp segment for a row of n relative positions.
__host__ __device__ __forceinline__ int rk_segment(int n) {
  return ((n + 32 * 128 - 1) / (32 * 128)) * 128;
}

__device__ __forceinline__ uint32_t rk_lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of one value per thread over the 1024-thread block; tmp
// holds 32 words.  Returns this thread's prefix; total = the block's sum.
__device__ __forceinline__ uint32_t rk_block_excl_scan(uint32_t v, uint32_t* tmp, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  uint32_t t = tmp[lane], incl = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t wbase = __shfl_sync(0xffffffffu, incl - t, warp);
  total = __shfl_sync(0xffffffffu, incl, 31);
  __syncthreads();
  return wbase + x - v;
}

// Radix select of the k-th largest key among the keys that `visit` feeds in.
// visit(f) calls f(key, live) for every key (each thread its own share, the
// same number of calls in every lane of a warp); dead keys, key 0 and keys
// whose bits above `top` differ from `prefix` are ignored.  The histogram has
// a private column per lane (bank = lane), so increments never collide inside
// a warp however skewed the digits are.  Returns T and need_eq.
template <class Visit>
__device__ __forceinline__ void rk_radix(Visit visit, int top, uint32_t prefix, uint32_t k,
                                         RowTopkSmem& sm, uint32_t& T, uint32_t& need_eq) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t mask = top >= 31 ? 0u : ~((2u << top) - 1u);
  prefix &= mask;
  uint32_t krem = k;
  uint4* h4 = reinterpret_cast<uint4*>(&sm.lhist[0][0]);
  for (int i = tid; i < 256 * 32 / 4; i += kRkThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
#pragma unroll 1
  for (int hi = top; hi >= 0; hi -= 8) {
    const int shift = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (2u << (hi - shift)) - 1u;
    visit([&](uint32_t u, bool live) {
      if (live && u != 0u && (u & mask) == prefix) atomicAdd(&sm.lhist[(u >> shift) & dmask][lane], 1u);
    });
    __syncthreads();
    {  // column sums: four threads per bin, eight lanes each
      const int bin = tid >> 2, q = (tid & 3) * 8;
      const uint4 x = *reinterpret_cast<const uint4*>(&sm.lhist[bin][q]);
      const uint4 y = *reinterpret_cast<const uint4*>(&sm.lhist[bin][q + 4]);
      uint32_t t = x.x + x.y + x.z + x.w + y.x + y.y + y.z + y.w;
      t += __shfl_xor_sync(0xffffffffu, t, 1);
      t += __shfl_xor_sync(0xffffffffu, t, 2);
      if ((tid & 3) == 0) sm.hist[bin] = t;
    }
    __syncthreads();
    for (int i = tid; i < 256 * 32 / 4; i += kRkThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
    // digit holding the krem-th largest, scanned from the top bin down
    if ((tid >> 5) == 0) {
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
    __syncthreads();
    krem -= sm.above;
    prefix |= sm.digit << shift;
    mask |= dmask << shift;
  }
  __syncthreads();
  T = prefix;
  need_eq = krem;
}

// A key whose rank among all keys is, with high probability, at least k and
// at most a few standard deviations above: the (est + margin)-th largest of a
// systematic sample of min(1024, n) keys, found by the same radix select.
template <class Src>
__device__ __forceinline__ uint32_t rk_sample_bound(const Src& src, int k, RowTopkSmem& sm) {
  const int tid = threadIdx.x;
  const int nvalid = src.n - src.lo;
  const int ns = min(kRkThreads, nvalid);
  const uint32_t mine = tid < ns ? src.load1(src.lo + int((long long)tid * nvalid / ns)) : 0u;
  const float p = float(k) / float(nvalid);
  const int est = int((long long)k * ns / nvalid);
  const int margin = 16 + int(4.0f * sqrtf(float(ns) * p * (1.f - p)));
  if (est + margin >= ns) return 1u;
  uint32_t t, unused;
  rk_radix([&](auto&& f) { f(mine, true); }, 31, 0u, uint32_t(est + margin + 1), sm, t, unused);
  return t > 1u ? t : 1u;
}

// Exact top-k over the row described by src (n = src.n relative positions,
// 1 <= k <= number of valid positions).  emit(i, rel) is called once for
// each kept position with its output index i in [0, k), indices ascending in
// rel.  hint: a lower bound to try first (0 = none).  Returns the k-th key T.
template <int kG, class Src, class Emit>
__device__ __forceinline__ uint32_t row_topk(const Src& src, int k, uint32_t hint, RowTopkSmem& sm,
                                             Emit emit) {
  constexpr int kR = 4 * kG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = rk_segment(src.n);
  const int ngroups = L / 128;
  const int wbase = warp * L;
  const bool resident = ngroups <= kG;
  uint32_t key[kR];
  auto load_chunk = [&](int g0) {
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (g0 + g < ngroups) v = src.load4(wbase + (g0 + g) * 128 + 4 * lane);
      key[4 * g] = v.x;
      key[4 * g + 1] = v.y;
      key[4 * g + 2] = v.z;
      key[4 * g + 3] = v.w;
    }
  };
  // sweep(f): f(g0) for every register chunk, keys loaded
  auto sweep = [&](auto&& f) {
    if (resident) {
      f(0);
    } else {
#pragma unroll 1
      for (int g0 = 0; g0 < ngroups; g0 += kG) {
        load_chunk(g0);
        f(g0);
      }
    }
  };
  if (resident) load_chunk(0);

  // --- 1-2. lower bound and the upper set ---------------------------------
  auto gather = [&](uint32_t t_lo) -> uint32_t {
    __syncthreads();
    if (tid == 0) {
      sm.cnt = 0;
      sm.maxkey = 0;
    }
    __syncthreads();
    uint32_t mx = 0;
    sweep([&](int) {
      uint32_t c = 0;
#pragma unroll
      for (int i = 0; i < kR; ++i) c += key[i] >= t_lo;
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t wsum = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t base = 0;
      if (lane == 31 && wsum) base = atomicAdd(&sm.cnt, wsum);
      base = __shfl_sync(0xffffffffu, base, 31) + incl - c;
#pragma unroll
      for (int i = 0; i < kR; ++i)
        if (key[i] >= t_lo) {
          if (base < uint32_t(kRkUpMax)) sm.ukey[base] = key[i];
          ++base;
          mx = max(mx, key[i]);
        }
    });
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0 && mx) atomicMax(&sm.maxkey, mx);
    __syncthreads();
    return sm.cnt;
  };
  uint32_t t_lo = hint, up_tot = 0;
  bool ok = false;
  if (t_lo != 0u) {
    up_tot = gather(t_lo);
    ok = up_tot >= uint32_t(k) && up_tot <= uint32_t(kRkUpMax);
  }
  if (!ok) {
    t_lo = rk_sample_bound(src, k, sm);
    up_tot = gather(t_lo);
    ok = up_tot >= uint32_t(k) && up_tot <= uint32_t(kRkUpMax);
  }

  // --- 3. the k-th key ----------------------------------------------------
  uint32_t T, need_eq;
  if (ok) {
    const uint32_t mx = sm.maxkey;
    const uint32_t diff = t_lo ^ mx;
    if (diff == 0u) {  // every key of the upper set equals t_lo
      T = t_lo;
      need_eq = uint32_t(k);
    } else {
      const int top = 31 - __clz(diff);
      const uint32_t up_round = (up_tot + 31u) & ~31u;
      rk_radix(
          [&](auto&& f) {
            for (uint32_t i = tid; i < up_round; i += kRkThreads) {
              const bool live = i < up_tot;
              f(live ? sm.ukey[i] : 0u, live);
            }
          },
          top, t_lo, uint32_t(k), sm, T, need_eq);
    }
  } else {
    rk_radix(
        [&](auto&& f) {
          sweep([&](int) {
#pragma unroll
            for (int i = 0; i < kR; ++i) f(key[i], true);
          });
        },
        31, 0u, uint32_t(k), sm, T, need_eq);
  }

  // --- 4. ordered emission ------------------------------------------------
  uint32_t gt = 0, eq = 0;
  sweep([&](int) {
#pragma unroll
    for (int i = 0; i < kR; ++i) {
      gt += key[i] > T;
      eq += key[i] == T;
    }
  });
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) {
    sm.wtot[0][warp] = gt;
    sm.wtot[1][warp] = eq;
  }
  __syncthreads();
  uint32_t g_in = sm.wtot[0][lane], e_in = sm.wtot[1][lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(0xffffffffu, g_in, o);
    const uint32_t b = __shfl_up_sync(0xffffffffu, e_in, o);
    if (lane >= o) {
      g_in += a;
      e_in += b;
    }
  }
  const uint32_t g_before = __shfl_sync(0xffffffffu, g_in, warp) - sm.wtot[0][warp];
  uint32_t eq_seen = __shfl_sync(0xffffffffu, e_in, warp) - sm.wtot[1][warp];
  uint32_t out = g_before + min(eq_seen, need_eq);
  const uint32_t lt = rk_lanemask_lt();
  const bool staged = k <= kRkUpMax;  // the upper set is no longer needed: stage the output there
  sweep([&](int g0) {
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      bool isgt[4], iseq[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        isgt[c] = key[4 * g + c] > T;
        iseq[c] = key[4 * g + c] == T;
      }
      // equal keys before this lane in this group (position order: lane-major)
      uint32_t eq_lane = 0, beq = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t b = __ballot_sync(0xffffffffu, iseq[c]);
        eq_lane += __popc(b & lt);
        beq += __popc(b);
      }
      uint32_t rank = eq_seen + eq_lane;
      bool keep[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        keep[c] = isgt[c] || (iseq[c] && rank < need_eq);
        rank += iseq[c];
      }
      uint32_t kept_lane = 0, kept_all = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t b = __ballot_sync(0xffffffffu, keep[c]);
        kept_lane += __popc(b & lt);
        kept_all += __popc(b);
      }
      uint32_t o = out + kept_lane;
      const int rel0 = wbase + (g0 + g) * 128 + 4 * lane;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (keep[c]) {
          if (o < uint32_t(k)) {  // never more than k, whatever the keys
            if (staged)
              sm.ukey[o] = uint32_t(rel0 + c);
            else
              emit(int(o), rel0 + c);
          }
          ++o;
        }
      out += kept_all;
      eq_seen += beq;
    }
  });
  if (staged) {  // the kept positions, in order, from shared memory: coalesced output writes
    __syncthreads();
    for (int i = tid; i < k; i += kRkThreads) emit(i, int(sm.ukey[i]));
  }
  return T;
}

}  // namespace kvsel
