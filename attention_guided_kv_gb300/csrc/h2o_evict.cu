// H2O heavy-hitter selection with StreamingLLM sinks + recent window, and
// order-preserving in-place compaction of the paged cache (sm_103a).
//
// What it computes ("From sliding window to attention-guided eviction" §4.1
// and the §4.2 pseudocode): per (sequence, kv head) with live length S >
// budget, keep slots [0, n_sink), the (budget - n_sink - window) slots of
// [n_sink, S - window) with the largest cumulative score (ties to the lower
// slot), and [S - window, S); evict the rest.
//
// select kernel, one 1024-thread CTA per (sequence, kv head):
//   finds the k-th largest score over the middle slots on a monotone uint32
//   image of the fp32 score.  The row's previous threshold (kept in the
//   workspace) usually bounds a band of about k keys from below; otherwise a
//   sorted sample brackets it; one counting pass gathers the keys inside the
//   band, and a 4 x 8-bit radix select finishes exactly (a radix select over
//   the whole row is the last fallback); then an
//   ordered emission: each thread owns a
//   contiguous run of slots, two block-wide scans give every thread its share
//   of the threshold ties (lowest slots first) and its output offset, so the
//   kept list comes out in ascending slot order without a sort.
// compact kernel, one CTA per (sequence, kv head): moves kept rows to slots
//   0..n_keep-1 in chunks of 64 slots.  Each chunk reads all of its sources
//   into shared memory before writing any destination; a kept list is sorted
//   and keep[i] >= i, so no chunk overwrites a row that a later chunk still
//   has to read.
// truncate kernel, one CTA per sequence: releases the pages past
//   ceil(n_keep / page_size) and publishes the new length.
#include "common.cuh"
#include "topk_block.cuh"

namespace kvsel {

constexpr int kHD = 128;
constexpr int kPg = 16;
constexpr int kSelThreads = 1024;
constexpr int kChunk = 64;
constexpr int kItems = 32;

struct SelectParams {
  const int32_t* seq_lens;
  const float* cum;
  const int32_t* pos_map;
  int32_t* keep_slots;  // workspace [B][Hkv][budget]
  int32_t* keep_out;    // [B][Hkv][budget] or null
  int32_t* first_move;  // workspace [B][Hkv]
  uint32_t* hint;       // workspace [B][Hkv]: last threshold key per row (0 = none)
  int* status;
  int Hkv, max_len, budget, n_sink, window;
};

// Per (sequence, kv head) row: the k kept middle slots (ties to the lower
// slot), ascending.  Register path (rows of at most kSelThreads * kItems
// candidates): each thread holds its contiguous run of candidate keys; the
// row's previous threshold (kept in the workspace), or else a sample
// quantile, bounds the k-th key from below and block_topk_upper finishes on
// the keys above that bound.  Last fallback (and longer rows): a radix select
// over the whole row in global memory, then an ordered emission over it.
template <bool kInRegs>
__global__ void __launch_bounds__(kSelThreads) h2o_select_kernel(const SelectParams P) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  UpperSmem& up = *reinterpret_cast<UpperSmem*>(sel_smem);
  __shared__ int s_first;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the scores come from the previous kernel

  const int kvh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  const int S = P.seq_lens[b];
  const size_t rowi = size_t(b) * P.Hkv + kvh;
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
    if (tid == 0) P.first_move[rowi] = S;
    return;
  }

  const int k = P.budget - P.n_sink - P.window;
  const int lo = P.n_sink, hi = S - P.window;
  const int n_cand = hi - lo;
  const int C = (n_cand + kSelThreads - 1) / kSelThreads;
  const int j0 = lo + min(n_cand, tid * C);
  const int cnt = min(n_cand, (tid + 1) * C) - min(n_cand, tid * C);
  uint32_t T = 0xFFFFFFFFu, need_eq = 0;
  bool done = false;
  if constexpr (kInRegs) {
    if (k > 0) {
      uint32_t key[kItems];
#pragma unroll
      for (int e = 0; e < kItems; ++e) key[e] = e < cnt ? order_key(row[j0 + e]) : 0u;
      auto pos_of = [&](int e) { return j0 + e; };
      const uint32_t hint = P.hint[rowi];
      done = block_topk_upper<kItems>(key, cnt, pos_of, n_cand, k, hint, up, keep + P.n_sink, T, need_eq);
      if (!done && hint != 0u)
        done = block_topk_upper<kItems>(key, cnt, pos_of, n_cand, k, 0u, up, keep + P.n_sink, T, need_eq);
    }
  }
  if (k > 0 && !done) {
    // whole-row radix select in global memory
    uint32_t prefix = 0, mask = 0, krem = uint32_t(k);
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) up.base.hist[tid] = 0;
      __syncthreads();
      for (int j = lo + tid; j < hi; j += kSelThreads) {
        const uint32_t u = order_key(row[j]);
        if ((u & mask) == prefix) atomicAdd(&up.base.hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      topk_pick_digit(up.base, krem);
      __syncthreads();
      krem -= up.base.above;
      prefix |= up.base.digit << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    T = prefix;
    need_eq = krem;
    // ordered emission over the whole row (contiguous runs per thread)
    uint32_t gt = 0, eq = 0;
    for (int e = 0; e < cnt; ++e) {
      const uint32_t u = order_key(row[j0 + e]);
      gt += u > T;
      eq += u == T;
    }
    uint32_t tot;
    const uint32_t eq_base = topk_block_scan(eq, up.base.scan, tot);
    const uint32_t take_eq = need_eq > eq_base ? min(eq, need_eq - eq_base) : 0u;
    uint32_t w = P.n_sink + topk_block_scan(gt + take_eq, up.base.scan, tot), q = eq_base;
    const uint32_t wend = uint32_t(P.n_sink + k);
    for (int e = 0; e < cnt; ++e) {
      const uint32_t u = order_key(row[j0 + e]);
      const bool isq = u == T;
      if ((u > T || (isq && q < need_eq)) && w < wend) keep[w++] = j0 + e;
      q += isq;
    }
  }
  if (k > 0 && tid == 0) P.hint[rowi] = T;
  for (int i = tid; i < P.n_sink; i += kSelThreads) keep[i] = i;
  for (int i = tid; i < P.window; i += kSelThreads) keep[P.budget - P.window + i] = S - P.window + i;
  if (tid == 0) s_first = P.budget;
  __syncthreads();
  int first = P.budget;
  for (int i = tid; i < P.budget; i += kSelThreads) {
    const int slot = keep[i];
    if (kout) kout[i] = prow ? prow[slot] : slot;
    if (slot != i) first = min(first, i);
  }
  atomicMin(&s_first, first);
  __syncthreads();
  if (tid == 0) P.first_move[rowi] = s_first;
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
};

__device__ __forceinline__ size_t pool_row(const int32_t* bt, int slot, int Hkv, int kvh,
                                           int num_pages, int* status, bool& ok) {
  const int phys = bt[slot / kPg];
  ok = unsigned(phys) < unsigned(num_pages);
  if (!ok) report(status, KVSEL_ERR_BAD_INDEX);
  return (size_t(phys) * Hkv + kvh) * kPg + (slot % kPg);
}

__global__ void __launch_bounds__(256) h2o_compact_kernel(const CompactParams P) {
  __shared__ uint4 sk[kChunk][16];
  __shared__ uint4 sv[kChunk][16];
  __shared__ float sc[kChunk];
  __shared__ int32_t sp[kChunk];
  const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int S = P.seq_lens[b];
  if (S <= P.budget) return;
  if (S > P.max_len || S > P.max_pages * kPg) {
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
      const size_t r = pool_row(bt, keep[c0 + t], P.Hkv, kvh, P.num_pages, P.status, ok);
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
      const size_t r = pool_row(bt, c0 + t, P.Hkv, kvh, P.num_pages, P.status, ok);
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
};

__global__ void __launch_bounds__(256) h2o_truncate_kernel(const TruncateParams P) {
  const int b = blockIdx.x;
  const int S = P.seq_lens[b];
  if (S > P.max_len) return;
  const int n_keep = S > P.budget ? P.budget : S;
  const int old_pages = min(P.max_pages, (S + kPg - 1) / kPg);
  const int new_pages = (n_keep + kPg - 1) / kPg;
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
  size_t keep_off, first_off, hint_off, total;
};
EvictWs evict_ws_layout(int batch, int Hkv, int budget) {
  EvictWs w;
  size_t off = kStatusBytes;
  w.keep_off = off;
  off = align_up(off + size_t(batch) * Hkv * budget * sizeof(int32_t), 256);
  w.first_off = off;
  off = align_up(off + size_t(batch) * Hkv * sizeof(int32_t), 256);
  w.hint_off = off;
  off = align_up(off + size_t(batch) * Hkv * sizeof(uint32_t), 256);
  w.total = off;
  return w;
}
}  // namespace

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
  if (kv->page_size != kPg || kv->head_dim != kHD)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16 are implemented");
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
  P.hint = reinterpret_cast<uint32_t*>(ws + L.hint_off);
  P.status = reinterpret_cast<int*>(ws);
  P.Hkv = kv->num_kv_heads;
  P.max_len = max_len;
  P.budget = budget;
  P.n_sink = n_sink;
  P.window = window;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kv->num_kv_heads, batch);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = kTopkDynSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool in_regs = (long long)max_len - n_sink - window <= (long long)kSelThreads * kItems;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t a1 = cudaFuncSetAttribute(h2o_select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTopkDynSmem));
    cudaError_t a2 = cudaFuncSetAttribute(h2o_select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTopkDynSmem));
    if (a1 != cudaSuccess || a2 != cudaSuccess) return cuda_fail(a1 != cudaSuccess ? a1 : a2, "kvsel_h2o_evict (attribute)");
    attr_set = true;
  }
  trace_before("h2o_select", st);
  cudaError_t e = in_regs ? cudaLaunchKernelEx(&cfg, h2o_select_kernel<true>, P)
                          : cudaLaunchKernelEx(&cfg, h2o_select_kernel<false>, P);
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
  trace_before("h2o_compact", st);
  h2o_compact_kernel<<<dim3(kv->num_kv_heads, batch), 256, 0, st>>>(C);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_h2o_evict (compact launch)");

  TruncateParams T;
  T.seq_lens = seq_lens;
  T.block_table = block_table;
  T.freed = freed_pages;
  T.max_pages = max_pages;
  T.budget = budget;
  T.max_len = max_len;
  trace_before("h2o_truncate", st);
  h2o_truncate_kernel<<<batch, 256, 0, st>>>(T);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_h2o_evict (truncate launch)");
  return KVSEL_OK;
}
