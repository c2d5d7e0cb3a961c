// H2O heavy-hitter selection with StreamingLLM sinks + recent window, and
// order-preserving in-place compaction of the paged cache (sm_103a).
//
// What it computes ("From sliding window to attention-guided eviction" §4.1
// and the §4.2 pseudocode): per (sequence, kv head) with live length S >
// budget, keep slots [0, n_sink), the (budget - n_sink - window) slots of
// [n_sink, S - window) with the largest cumulative score (ties to the lower
// slot), and [S - window, S); evict the rest.
//
// select kernel, one 1024-thread CTA per (sequence, kv head): an exact
//   top-k over a monotone uint32 image of the fp32 score (row_topk.cuh):
//   coalesced float4 loads into registers, a lower bound on the k-th key
//   (the row's previous threshold, kept in the workspace, else a sample
//   quantile), a radix select over the keys above that bound only, and an
//   ordered emission that writes the kept list in ascending slot order
//   (lowest slots first among ties) without a sort.
// compact kernel, one CTA per (sequence, kv head): moves kept rows to slots
//   0..n_keep-1 in chunks of 64 slots.  Each chunk reads all of its sources
//   into shared memory before writing any destination; a kept list is sorted
//   and keep[i] >= i, so no chunk overwrites a row that a later chunk still
//   has to read.
// truncate kernel, one CTA per sequence: releases the pages past
//   ceil(n_keep / page_size) and publishes the new length.
#include "common.cuh"
#include "h2o_link.cuh"
#include "row_topk.cuh"

namespace kvsel {

constexpr int kHD = 128;
constexpr int kPg = 16;  // the smallest page; pools may use 16 << page_shift tokens per page
constexpr int kSelThreads = 1024;
constexpr int kChunk = 64;
constexpr int kSelGroups = 8;  // register-resident rows: up to 32 x 8 x 128 candidates

struct SelectParams {
  const int32_t* seq_lens;
  const float* cum;
  const int32_t* pos_map;
  int32_t* keep_slots;  // workspace [B][Hkv][budget]
  int32_t* keep_out;    // [B][Hkv][budget] or null
  int32_t* first_move;  // workspace [B][Hkv]
  H2OLink link;         // workspace: thresholds and the decode step's candidate lists
  int* status;
  int Hkv, max_len, budget, n_sink, window;
};

constexpr int kListWords = 1024;  // list path: rows of up to 32768 candidate slots

struct SelSmem {
  RowTopkSmem rk;
  int32_t upos[kRkUpMax];           // listed slots (then relative to the candidate range)
  uint32_t bits[2][kListWords];     // kept-above / tie bitmaps over the candidate slots
  uint32_t m, minkey, bad;
  uint64_t bar;                     // completion of the list's bulk copy
};
static_assert(kRkUpMax >= kLinkCap, "every listed slot fits in shared memory");
static_assert(offsetof(RowTopkSmem, ukey) % 16 == 0 && offsetof(SelSmem, upos) % 16 == 0,
              "bulk copies land on 16-byte boundaries");

__device__ __forceinline__ uint32_t lowest_bits(uint32_t x, uint32_t n) {
  uint32_t r = 0;
  for (uint32_t t = 0; t < n && x; ++t) {
    const uint32_t b = x & (0u - x);
    r |= b;
    x ^= b;
  }
  return r;
}

// Radix select of the k-th largest of the live keys ukey[0..cnt) (key 0: not a
// candidate; keys whose bits above `top` differ from `prefix` are ignored)
// with 11-bit digits from bit `top` down, so a 32-bit spread takes three
// passes.  A candidate list is small, so one shared histogram of 2048 bins
// takes the increments directly; two histograms alternate, each pass clearing
// the next one's.  The bins are scanned from the top down, two per thread.
// Returns T and need_eq (how many keys equal to T are kept).
__device__ __forceinline__ void list_radix(const uint32_t* ukey, uint32_t cnt, int top, uint32_t prefix, uint32_t k,
                                           RowTopkSmem& rk, uint32_t& T, uint32_t& need_eq) {
  static_assert(sizeof(RowTopkSmem::lhist) >= 2 * 2048 * sizeof(uint32_t), "two histograms of 2048 bins");
  static_assert(kSelThreads * 2 == 2048, "two bins per thread");
  const int tid = threadIdx.x;
  uint32_t* H = &rk.lhist[0][0];
  uint32_t mask = top >= 31 ? 0u : ~((2u << top) - 1u);
  prefix &= mask;
  uint32_t krem = k;
  for (int i = tid; i < 2048; i += kSelThreads) H[i] = 0u;
  __syncthreads();
#pragma unroll 1
  for (int hi = top, pass = 0; hi >= 0; hi -= 11, ++pass) {
    uint32_t* h = H + (pass & 1) * 2048;
    uint32_t* hn = H + ((pass + 1) & 1) * 2048;
    const int shift = hi >= 10 ? hi - 10 : 0;
    const uint32_t dmask = (2u << (hi - shift)) - 1u;
    for (uint32_t i = tid; i < cnt; i += kSelThreads) {
      const uint32_t u = ukey[i];
      if (u != 0u && (u & mask) == prefix) atomicAdd(&h[(u >> shift) & dmask], 1u);
    }
    for (int i = tid; i < 2048; i += kSelThreads) hn[i] = 0u;
    __syncthreads();
    const uint32_t c0 = h[2047 - 2 * tid], c1 = h[2046 - 2 * tid];
    uint32_t tot;
    const uint32_t ex = rk_block_excl_scan(c0 + c1, rk.wtot[0], tot);
    if (ex < krem && krem <= ex + c0 + c1) {  // this thread's bins hold the krem-th largest
      const bool first = krem <= ex + c0;
      rk.digit = first ? 2047u - 2u * tid : 2046u - 2u * tid;
      rk.above = first ? ex : ex + c0;
    }
    __syncthreads();
    krem -= rk.above;
    prefix |= rk.digit << shift;
    mask |= dmask << shift;
  }
  T = prefix;
  need_eq = krem;
}

// Top-k of the middle slots [lo, hi) from the candidate list that the decode
// step collected (every slot whose score is >= the row's last threshold).
// Usable when the list is fresh and holds at least k slots of [lo, hi): the
// k-th score is then >= the old threshold, so the list holds every slot the
// top k can contain.  Freshness is checked on the first 1024 entries (their
// listed score must still equal the row's score at that slot); any later
// decode step changes every listed score, since each live slot gains a
// positive probability.  Emits the kept slots through put(i, slot) in ascending
// order and returns true, else returns false (block-uniform) having written
// nothing.
template <class Put>
__device__ __forceinline__ bool select_from_list(const SelectParams& P, size_t rowi, const float* row,
                                                 uint32_t cnt, int lo, int hi, int k, SelSmem& sm,
                                                 uint32_t& T, Put put) {
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t* lk = P.link.key + rowi * kLinkCap;
  const int32_t* lp = P.link.pos + rowi * kLinkCap;
  const int nw = (hi - lo + 31) >> 5;
  const uint32_t bar = smem_u32(&sm.bar);
  if (tid == 0) {
    sm.m = 0;
    sm.rk.maxkey = 0;
    sm.minkey = 0xFFFFFFFFu;
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  for (int i = tid; i < nw; i += kSelThreads) sm.bits[0][i] = sm.bits[1][i] = 0u;
  __syncthreads();
  if (tid == 0) {  // the whole list into shared memory: two bulk copies (rows are 64 KB apart)
    const uint32_t bytes = (cnt * 4u + 15u) & ~15u;
    mbar_expect_tx(bar, 2u * bytes);
    bulk_load(smem_u32(sm.rk.ukey), lk, bytes, bar);
    bulk_load(smem_u32(sm.upos), lp, bytes, bar);
  }
  // freshness, while the copies run: the first listed scores must still be the row's
  uint32_t bad = 0;
  if (uint32_t(tid) < cnt) {
    const uint32_t key = __ldcg(lk + tid);
    const int pos = __ldcg(lp + tid);
    if (pos < 0 || pos >= P.max_len) bad = 1;
    else bad |= order_key(__ldcg(row + pos)) != key;
  }
  if (!mbar_wait(bar, 0u, P.status)) bad = 1;
  // one sweep: entries outside [lo, hi) get key 0 (skipped from here on), the
  // others their slot relative to lo; count, smallest and largest key
  uint32_t mx = 0, mn = 0xFFFFFFFFu, n_in = 0;
  for (uint32_t i = tid; i < cnt; i += kSelThreads) {
    const uint32_t key = sm.rk.ukey[i];
    const int pos = sm.upos[i];
    if (pos < 0 || pos >= P.max_len) bad = 1;
    if (pos >= lo && pos < hi) {
      sm.upos[i] = pos - lo;
      mx = max(mx, key);
      mn = min(mn, key);
      ++n_in;
    } else {
      sm.rk.ukey[i] = 0u;
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  n_in = __reduce_add_sync(0xffffffffu, n_in);
  if (lane == 0) {
    if (mx) atomicMax(&sm.rk.maxkey, mx);
    atomicMin(&sm.minkey, mn);
    atomicAdd(&sm.m, n_in);
  }
  if (__syncthreads_or(bad)) return false;
  const uint32_t m = sm.m;
  if (m < uint32_t(k)) return false;
  uint32_t need_eq;
  const uint32_t lo_key = sm.minkey, hi_key = sm.rk.maxkey;
  if (lo_key == hi_key) {
    T = lo_key;
    need_eq = uint32_t(k);
  } else {
    list_radix(sm.rk.ukey, cnt, 31 - __clz(lo_key ^ hi_key), lo_key, uint32_t(k), sm.rk, T, need_eq);
  }
  for (uint32_t i = tid; i < cnt; i += kSelThreads) {
    const uint32_t u = sm.rk.ukey[i];
    if (u == 0u) continue;  // outside the candidate range
    const int r = sm.upos[i];
    if (u > T) atomicOr(&sm.bits[0][r >> 5], 1u << (r & 31));
    else if (u == T) atomicOr(&sm.bits[1][r >> 5], 1u << (r & 31));
  }
  __syncthreads();
  // ordered emission: thread t owns bitmap word t (32 slots)
  const uint32_t wg = tid < nw ? sm.bits[0][tid] : 0u, we = tid < nw ? sm.bits[1][tid] : 0u;
  uint32_t total;
  const uint32_t ex = rk_block_excl_scan(uint32_t(__popc(wg)) | (uint32_t(__popc(we)) << 16), sm.rk.wtot[0], total);
  const uint32_t g_before = ex & 0xFFFFu, e_before = ex >> 16;
  const uint32_t take = need_eq > e_before ? min(uint32_t(__popc(we)), need_eq - e_before) : 0u;
  uint32_t keepw = wg | lowest_bits(we, take);
  uint32_t o = g_before + min(e_before, need_eq);
  uint32_t* staged = sm.rk.ukey;
  while (keepw) {
    const int bit = __ffs(keepw) - 1;
    keepw &= keepw - 1;
    if (o < uint32_t(k)) staged[o] = uint32_t(tid * 32 + bit);
    ++o;
  }
  __syncthreads();
  for (int i = tid; i < k; i += kSelThreads) put(i, lo + int(staged[i]));
  return true;
}

// Per (sequence, kv head) row: the sinks, the k heaviest middle slots
// [n_sink, S - window) (ties to the lower slot) and the window, ascending.
// row_topk selects the middle slots, trying the row's previous threshold
// (kept in the workspace) as its first lower bound; the kept list, the
// original positions and the first slot that moves are written as the
// positions are emitted.
__global__ void __launch_bounds__(kSelThreads) h2o_select_kernel(const SelectParams P) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(sel_smem);
  __shared__ int s_first;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the scores come from the previous kernel
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  const size_t rowi = size_t(b) * P.Hkv + kvh;
  // the length, the decode step's candidate count and the row's last
  // threshold, in one round trip
  const int S = P.seq_lens[b];
  const uint32_t cnt = __ldcg(P.link.count + rowi);
  const uint32_t hk = __ldcg(P.link.hint + rowi);
  // A decode step launched after this kernel may start now: it publishes new
  // lengths early (read above), and touches the scores, the candidate lists
  // and the thresholds only after waiting for this kernel to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float* row = P.cum + rowi * P.max_len;
  const int32_t* prow = P.pos_map ? P.pos_map + rowi * P.max_len : nullptr;
  int32_t* keep = P.keep_slots + rowi * P.budget;
  int32_t* kout = P.keep_out ? P.keep_out + rowi * P.budget : nullptr;

  if (S < 0 || S > P.max_len) {
    if (tid == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  if (S <= P.budget) {
    for (int i = tid; i < P.budget; i += kSelThreads) {
      const int slot = i < S ? i : -1;
      keep[i] = slot;
      if (kout) kout[i] = slot < 0 ? -1 : (prow ? prow[slot] : slot);
    }
    if (tid == 0) {
      P.first_move[rowi] = S;
      P.link.count[rowi] = 0u;  // a list is used at most once
    }
    return;
  }
  if (tid == 0) s_first = P.budget;
  __syncthreads();

  const int k = P.budget - P.n_sink - P.window;
  int first = P.budget;
  auto put = [&](int o, int slot) {
    keep[o] = slot;
    if (kout) kout[o] = prow ? prow[slot] : slot;
    if (slot != o) first = min(first, o);
  };
  // the sinks and the window do not depend on the selection: written first
  for (int i = tid; i < P.n_sink; i += kSelThreads) put(i, i);
  for (int i = tid; i < P.window; i += kSelThreads) put(P.budget - P.window + i, S - P.window + i);
  if (k > 0) {
    const int lo = P.n_sink, hi = S - P.window;
    uint32_t T = 0;
    bool done = false;
    if (hk != 0u && cnt >= uint32_t(k) && cnt <= uint32_t(kLinkCap) && hi - lo <= 32 * kListWords)
      done = select_from_list(P, rowi, row, cnt, lo, hi, k, sm, T,
                              [&](int i, int slot) { put(P.n_sink + i, slot); });
    if (!done) {
      const int a = P.n_sink & ~3;  // float4-aligned start of the candidate run
      const float* base = row + a;
      const F32RowKeys src{base, P.n_sink - a, S - P.window - a,
                           (reinterpret_cast<uintptr_t>(base) & 15u) == 0};
      T = row_topk<kSelGroups>(src, k, hk, sm.rk, [&](int i, int rel) { put(P.n_sink + i, a + rel); });
    }
    if (tid == 0) P.link.hint[rowi] = T;
  }
  if (first < P.budget) atomicMin(&s_first, first);
  __syncthreads();
  if (tid == 0) {
    P.first_move[rowi] = s_first;
    P.link.count[rowi] = 0u;
  }
}

struct CompactParams {
  const int32_t* seq_lens;
  const int32_t* block_table;
  const int32_t* keep_slots;
  const int32_t* first_move;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  float* cum;
  int32_t* pos_map;
  int* status;
  int Hkv, max_len, max_pages, num_pages, budget;
  int page_shift;  // log2(page_size / 16)
};

// Pool row of a sequence's slot: page block_table[slot / page_size], row
// slot % page_size of the kv head's part of that page.
__device__ __forceinline__ size_t pool_row(const int32_t* bt, int slot, int Hkv, int kvh, int page_shift,
                                           int num_pages, int* status, bool& ok) {
  const int lg = 4 + page_shift;
  const int phys = bt[slot >> lg];
  ok = unsigned(phys) < unsigned(num_pages);
  if (!ok) report(status, KVSEL_ERR_BAD_INDEX);
  return ((size_t(phys) * Hkv + kvh) << lg) + (slot & ((1 << lg) - 1));
}

__global__ void __launch_bounds__(256) h2o_compact_kernel(const CompactParams P) {
  __shared__ uint4 sk[kChunk][16];
  __shared__ uint4 sv[kChunk][16];
  __shared__ float sc[kChunk];
  __shared__ int32_t sp[kChunk];
  const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  // launched early (programmatic serialization): the kept lists come from the select
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the truncation waits for this kernel
  const int S = P.seq_lens[b];
  if (S <= P.budget) return;
  if (S > P.max_len || (long long)S > ((long long)P.max_pages << (4 + P.page_shift))) {
    if (tid == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  const size_t rowi = size_t(b) * P.Hkv + kvh;
  const int32_t* keep = P.keep_slots + rowi * P.budget;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  float* crow = P.cum + rowi * P.max_len;
  int32_t* prow = P.pos_map ? P.pos_map + rowi * P.max_len : nullptr;
  const int n_keep = P.budget;
  const int t16 = tid & 15, tok = tid >> 4;  // 16 threads x 16 B per 256-byte row
#pragma unroll 1
  for (int c0 = P.first_move[rowi]; c0 < n_keep; c0 += kChunk) {
    const int cnt = min(kChunk, n_keep - c0);
    for (int t = tok; t < cnt; t += 16) {
      bool ok;
      const size_t r = pool_row(bt, keep[c0 + t], P.Hkv, kvh, P.page_shift, P.num_pages, P.status, ok);
      sk[t][t16] = ok ? reinterpret_cast<const uint4*>(P.k_pool + r * kHD)[t16] : make_uint4(0, 0, 0, 0);
      sv[t][t16] = ok ? reinterpret_cast<const uint4*>(P.v_pool + r * kHD)[t16] : make_uint4(0, 0, 0, 0);
    }
    if (tid < cnt) {
      const int src = keep[c0 + tid];
      sc[tid] = crow[src];
      if (prow) sp[tid] = prow[src];
    }
    __syncthreads();
    for (int t = tok; t < cnt; t += 16) {
      bool ok;
      const size_t r = pool_row(bt, c0 + t, P.Hkv, kvh, P.page_shift, P.num_pages, P.status, ok);
      if (ok) {
        reinterpret_cast<uint4*>(P.k_pool + r * kHD)[t16] = sk[t][t16];
        reinterpret_cast<uint4*>(P.v_pool + r * kHD)[t16] = sv[t][t16];
      }
    }
    if (tid < cnt) {
      crow[c0 + tid] = sc[tid];
      if (prow) prow[c0 + tid] = sp[tid];
    }
    __syncthreads();
  }
}

struct TruncateParams {
  int32_t* seq_lens;
  int32_t* block_table;
  int32_t* freed;
  int max_pages, budget, max_len;
  int page_shift;
};

__global__ void __launch_bounds__(256) h2o_truncate_kernel(const TruncateParams P) {
  const int b = blockIdx.x;
  // launched early (programmatic serialization): runs once the compaction is
  // done.  It does not let the next kernel start early: a decode step reads
  // the lengths and block table written here.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int S = P.seq_lens[b];
  if (S > P.max_len) return;
  const int n_keep = S > P.budget ? P.budget : S;
  const int psz = kPg << P.page_shift;
  const int old_pages = min(P.max_pages, (S + psz - 1) / psz);
  const int new_pages = (n_keep + psz - 1) / psz;
  int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  int32_t* fr = P.freed ? P.freed + size_t(b) * P.max_pages : nullptr;
  for (int p = threadIdx.x; p < P.max_pages; p += blockDim.x) {
    if (fr) fr[p] = (new_pages + p < old_pages) ? bt[new_pages + p] : -1;
  }
  __syncthreads();
  for (int p = new_pages + threadIdx.x; p < old_pages; p += blockDim.x) bt[p] = -1;
  if (threadIdx.x == 0) P.seq_lens[b] = n_keep;
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct EvictWs {
  size_t keep_off, first_off, total;
};
EvictWs evict_ws_layout(int batch, int Hkv, int budget) {
  EvictWs w;
  size_t off = link_bytes(batch * Hkv);  // status block + the decode hand-off (h2o_link.cuh)
  w.keep_off = off;
  off = align_up(off + size_t(batch) * Hkv * budget * sizeof(int32_t), 256);
  w.first_off = off;
  off = align_up(off + size_t(batch) * Hkv * sizeof(int32_t), 256);
  w.total = off;
  return w;
}
}  // namespace

extern "C" kvsel_status kvsel_h2o_link_reset(void* workspace, int batch, int num_kv_heads, void* stream) {
  const std::string fn = "kvsel_h2o_link_reset: ";
  if (!workspace || !aligned(workspace, 256) || batch < 1 || num_kv_heads < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "a 256-byte aligned workspace, batch >= 1 and num_kv_heads >= 1 are required");
  // the thresholds and the candidate counts (adjacent): no threshold, no list
  const H2OLink L = link_layout(workspace, batch * num_kv_heads);
  const size_t bytes = reinterpret_cast<uint8_t*>(L.key) - reinterpret_cast<uint8_t*>(L.hint);
  cudaError_t e = cudaMemsetAsync(L.hint, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_h2o_link_reset");
  return KVSEL_OK;
}

extern "C" size_t kvsel_h2o_link_bytes(int batch, int num_kv_heads) {
  if (batch < 1 || num_kv_heads < 1) return 0;
  return link_bytes(batch * num_kv_heads);
}

extern "C" size_t kvsel_h2o_evict_workspace(const kvsel_paged_kv* kv, int batch, int budget) {
  if (!kv || batch < 1 || budget < 1 || kv->num_kv_heads < 1) return 0;
  return evict_ws_layout(batch, kv->num_kv_heads, budget).total;
}

extern "C" kvsel_status kvsel_h2o_evict(const kvsel_paged_kv* kv, int32_t* block_table, int max_pages,
                                        int32_t* seq_lens, int batch, float* h2o_cum, int32_t* pos_map,
                                        int max_len, int budget, int n_sink, int window, int compact,
                                        int32_t* keep_out, int32_t* freed_pages, void* workspace,
                                        size_t ws_bytes, void* stream) {
  const std::string fn = "kvsel_h2o_evict: ";
  if (!kv || kv->num_kv_heads < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv descriptor is required");
  if (page_shift_of(kv->page_size) < 0 || kv->head_dim != kHD)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16, 32, 64, 128 or 256 are implemented");
  if (!block_table || !seq_lens || !h2o_cum || batch < 1 || max_pages < 1 || max_len < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "block_table, seq_lens, h2o_cum required; batch, max_pages, max_len >= 1");
  if (budget < 1 || n_sink < 0 || window < 0 || (long long)n_sink + window > budget)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "need budget >= 1, n_sink >= 0, window >= 0, n_sink + window <= budget");
  if (compact && (!kv->k_pool || !kv->v_pool))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "compaction needs the K and V pools");
  if (compact && (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16)))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pools must be 16-byte aligned");
  if (!workspace || !aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "a 256-byte aligned workspace is required");
  const EvictWs L = evict_ws_layout(batch, kv->num_kv_heads, budget);
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(L.total));

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SelectParams P;
  P.seq_lens = seq_lens;
  P.cum = h2o_cum;
  P.pos_map = pos_map;
  P.keep_slots = reinterpret_cast<int32_t*>(ws + L.keep_off);
  P.keep_out = keep_out;
  P.first_move = reinterpret_cast<int32_t*>(ws + L.first_off);
  P.link = link_layout(workspace, batch * kv->num_kv_heads);
  P.status = reinterpret_cast<int*>(ws);
  P.Hkv = kv->num_kv_heads;
  P.max_len = max_len;
  P.budget = budget;
  P.n_sink = n_sink;
  P.window = window;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kv->num_kv_heads, batch);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = sizeof(SelSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaError_t a = smem_limit_once(reinterpret_cast<const void*>(h2o_select_kernel), int(sizeof(SelSmem)));
      a != cudaSuccess)
    return cuda_fail(a, "kvsel_h2o_evict (attribute)");
  trace_before("h2o_select", st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, h2o_select_kernel, P);
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_h2o_evict (select launch)");
  if (!compact) return KVSEL_OK;

  CompactParams C;
  C.seq_lens = seq_lens;
  C.block_table = block_table;
  C.keep_slots = P.keep_slots;
  C.first_move = P.first_move;
  C.k_pool = static_cast<__nv_bfloat16*>(kv->k_pool);
  C.v_pool = static_cast<__nv_bfloat16*>(kv->v_pool);
  C.cum = h2o_cum;
  C.pos_map = pos_map;
  C.status = P.status;
  C.Hkv = kv->num_kv_heads;
  C.max_len = max_len;
  C.max_pages = max_pages;
  C.num_pages = kv->num_pages;
  C.budget = budget;
  C.page_shift = page_shift_of(kv->page_size);
  trace_before("h2o_compact", st);
  cfg.gridDim = dim3(kv->num_kv_heads, batch);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, h2o_compact_kernel, C);  // programmatic serialization, like the select
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_h2o_evict (compact launch)");

  TruncateParams T;
  T.seq_lens = seq_lens;
  T.block_table = block_table;
  T.freed = freed_pages;
  T.max_pages = max_pages;
  T.budget = budget;
  T.max_len = max_len;
  T.page_shift = C.page_shift;
  trace_before("h2o_truncate", st);
  cfg.gridDim = dim3(batch);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, h2o_truncate_kernel, T);
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_h2o_evict (truncate launch)");
  return KVSEL_OK;
}
