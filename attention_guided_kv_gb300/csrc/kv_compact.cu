// Keep-list compaction of the paged cache (sm_103a): after a selection, the
// kept K/V rows of every (sequence, kv head) move to slots 0..n-1 in order,
// the pages past ceil(n / page_size) are released and the length becomes n.
//
// What it computes ("From sliding window to attention-guided eviction":
// §4.2's pseudocode evicts every slot outside the keep set, and §4.3 step 6
// continues generation with only the kept KV): for keep row r (strictly
// ascending slots, all < S), slot i <- slot r[i] for i < n, for K, V and the
// optional per-slot score and position rows.
//
// check kernel, one CTA per sequence: validates every keep row of the
//   sequence (count, range, strict order; one count for all kv heads, since
//   one block table serves them) and finds each row's first slot that moves.
//   An invalid sequence is recorded as KVSEL_ERR_BAD_INDEX and left alone.
// move kernel, one CTA per (sequence, kv head): copies the rows in chunks of
//   128 slots, all of a chunk's sources read into registers before any of
//   its destinations is written (a block barrier between the two).  Rows are
//   strictly ascending, so r[i] >= i: a chunk writes only slots below every
//   source of the chunks after it, and the chunks run in order, so no source
//   is overwritten before it is read.
// truncate kernel, one CTA per sequence: lists and clears the released
//   block-table entries and publishes the new length.
#include "common.cuh"

namespace kvsel {

constexpr int kKcHD = 128;
constexpr int kKcPg = 16;         // the smallest page; pools may use 16 << page_shift tokens per page
constexpr int kKcChunk = 128;     // slots per chunk: 128 x 512 B of K and V held in registers
constexpr int kKcThreads = 512;
constexpr int kKcCheckThreads = 256;

struct KcParams {
  int32_t* seq_lens;
  int32_t* block_table;
  const int32_t* keep;
  const int32_t* keep_count;  // or null: a row's count is its run of entries >= 0
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  float* scores;              // [batch][Hkv][max_len] or null
  int32_t* pos_map;           // [batch][Hkv][max_len] or null
  int32_t* freed;             // [batch][max_pages] or null
  int32_t* n_keep;            // workspace [batch]: the sequence's count, -1 if rejected
  int32_t* first_move;        // workspace [batch][Hkv]
  int* status;
  int Hkv, keep_stride, max_len, max_pages, num_pages;
  int page_shift;             // log2(page_size / 16)
};

__global__ void __launch_bounds__(kKcCheckThreads) kc_check_kernel(const KcParams P) {
  // the move kernel may launch now; it waits for this grid at entry
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int s_n, s_bad, s_first;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int S = P.seq_lens[b];
  bool bad = S < 0 || (long long)S > ((long long)P.max_pages << (4 + P.page_shift)) ||
             ((P.scores || P.pos_map) && S > P.max_len);
  int n_all = -1;
  for (int g = 0; g < P.Hkv && !bad; ++g) {
    const size_t rowi = size_t(b) * P.Hkv + g;
    const int32_t* row = P.keep + rowi * P.keep_stride;
    if (tid == 0) {
      s_n = P.keep_stride;
      s_bad = 0;
      s_first = 0x7fffffff;
    }
    __syncthreads();
    int n;
    if (P.keep_count) {
      n = P.keep_count[rowi];
    } else {
      int first_neg = P.keep_stride;
      for (int i = tid; i < P.keep_stride; i += kKcCheckThreads)
        if (row[i] < 0) {
          first_neg = i;
          break;
        }
      if (first_neg < P.keep_stride) atomicMin(&s_n, first_neg);
      __syncthreads();
      n = s_n;
    }
    const bool n_ok = n >= 0 && n <= P.keep_stride && n <= S;
    int rb = 0, first = 0x7fffffff;
    if (n_ok) {
      for (int i = tid; i < n; i += kKcCheckThreads) {
        const int v = row[i];
        if (v < 0 || v >= S || (i > 0 && row[i - 1] >= v)) rb = 1;
        if (v != i) first = min(first, i);
      }
    }
    if (rb) atomicOr(&s_bad, 1);
    if (first != 0x7fffffff) atomicMin(&s_first, first);
    __syncthreads();
    bad = !n_ok || s_bad != 0 || (n_all >= 0 && n != n_all);
    n_all = n;
    if (tid == 0 && !bad) P.first_move[rowi] = min(s_first, n);
    __syncthreads();
  }
  if (tid == 0) {
    if (bad) report(P.status, KVSEL_ERR_BAD_INDEX);
    P.n_keep[b] = bad ? -1 : (P.Hkv > 0 ? n_all : 0);
  }
}

// Pool row of slot `slot` of kv head `kvh` through the sequence's block table:
// page block_table[slot / page_size], row slot % page_size of the head's part.
__device__ __forceinline__ size_t kc_pool_row(const int32_t* bt, int slot, int Hkv, int kvh, int page_shift,
                                              int num_pages, int* status, bool& ok) {
  const int lg = 4 + page_shift;
  const int phys = bt[slot >> lg];
  ok = unsigned(phys) < unsigned(num_pages);
  if (!ok) report(status, KVSEL_ERR_BAD_INDEX);
  return ((size_t(phys) * Hkv + kvh) << lg) + (slot & ((1 << lg) - 1));
}

constexpr int kKcRowsPerThread = kKcChunk / (kKcThreads / 16);

__global__ void __launch_bounds__(kKcThreads) kc_move_kernel(const KcParams P) {
  __shared__ int32_t s_src[kKcChunk];
  asm volatile("griddepcontrol.wait;" ::: "memory");                // counts and first moves
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the truncation waits for this grid
  const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int n = P.n_keep[b];
  if (n < 0) return;
  const size_t rowi = size_t(b) * P.Hkv + kvh;
  const int32_t* keep = P.keep + rowi * P.keep_stride;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  float* crow = P.scores ? P.scores + rowi * P.max_len : nullptr;
  int32_t* prow = P.pos_map ? P.pos_map + rowi * P.max_len : nullptr;
  const int part = tid & 15, r0 = tid >> 4;  // 16 threads x 16 B per 256-byte row
#pragma unroll 1
  for (int c0 = P.first_move[rowi]; c0 < n; c0 += kKcChunk) {
    const int cnt = min(kKcChunk, n - c0);
    if (tid < cnt) s_src[tid] = keep[c0 + tid];
    __syncthreads();
    // every source of the chunk into registers before any destination is written
    uint4 rk[kKcRowsPerThread], rv[kKcRowsPerThread];
#pragma unroll
    for (int j = 0; j < kKcRowsPerThread; ++j) {
      const int t = r0 + j * (kKcThreads / 16);
      rk[j] = rv[j] = make_uint4(0, 0, 0, 0);
      if (t < cnt) {
        bool ok;
        const size_t r = kc_pool_row(bt, s_src[t], P.Hkv, kvh, P.page_shift, P.num_pages, P.status, ok);
        if (ok) {
          rk[j] = __ldcs(reinterpret_cast<const uint4*>(P.k_pool + r * kKcHD) + part);
          rv[j] = __ldcs(reinterpret_cast<const uint4*>(P.v_pool + r * kKcHD) + part);
        }
      }
    }
    float sc = 0.f;
    int32_t ps = 0;
    if (tid < cnt) {
      if (crow) sc = crow[s_src[tid]];
      if (prow) ps = prow[s_src[tid]];
    }
    __syncthreads();  // every read of the chunk happens before any of its writes
#pragma unroll
    for (int j = 0; j < kKcRowsPerThread; ++j) {
      const int t = r0 + j * (kKcThreads / 16);
      if (t < cnt) {
        bool ok;
        const size_t r = kc_pool_row(bt, c0 + t, P.Hkv, kvh, P.page_shift, P.num_pages, P.status, ok);
        if (ok) {
          reinterpret_cast<uint4*>(P.k_pool + r * kKcHD)[part] = rk[j];
          reinterpret_cast<uint4*>(P.v_pool + r * kKcHD)[part] = rv[j];
        }
      }
    }
    if (tid < cnt) {
      if (crow) crow[c0 + tid] = sc;
      if (prow) prow[c0 + tid] = ps;
    }
    __syncthreads();  // the chunk's writes precede the next chunk's reads (s_src reuse too)
  }
}

__global__ void __launch_bounds__(kKcCheckThreads) kc_truncate_kernel(const KcParams P) {
  // runs once every move of the batch is done; the next kernel reads the
  // lengths and block table written here, so it is not let in early
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x;
  const int n = P.n_keep[b];
  if (n < 0) return;
  const int S = P.seq_lens[b];
  const int psz = kKcPg << P.page_shift;
  const int old_pages = (S + psz - 1) / psz;  // <= max_pages (checked)
  const int new_pages = (n + psz - 1) / psz;
  int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  if (P.freed) {
    int32_t* fr = P.freed + size_t(b) * P.max_pages;
    for (int p = threadIdx.x; p < P.max_pages; p += blockDim.x)
      fr[p] = (new_pages + p < old_pages) ? bt[new_pages + p] : -1;
  }
  __syncthreads();
  for (int p = new_pages + threadIdx.x; p < old_pages; p += blockDim.x) bt[p] = -1;
  if (threadIdx.x == 0) P.seq_lens[b] = n;
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct KcWs {
  size_t n_off, first_off, total;
};
KcWs kc_ws_layout(int batch, int Hkv) {
  KcWs w;
  w.n_off = kStatusBytes;
  w.first_off = align_up(w.n_off + size_t(batch) * sizeof(int32_t), 256);
  w.total = align_up(w.first_off + size_t(batch) * Hkv * sizeof(int32_t), 256);
  return w;
}
}  // namespace

extern "C" size_t kvsel_kv_compact_workspace(int batch, int num_kv_heads) {
  if (batch < 1 || num_kv_heads < 1) return 0;
  return kc_ws_layout(batch, num_kv_heads).total;
}

extern "C" kvsel_status kvsel_kv_compact(const kvsel_paged_kv* kv, int32_t* block_table, int max_pages,
                                         int32_t* seq_lens, int batch, const int32_t* keep, int keep_stride,
                                         const int32_t* keep_count, float* scores, int32_t* pos_map,
                                         int max_len, int32_t* freed_pages, void* workspace, size_t ws_bytes,
                                         void* stream) {
  const std::string fn = "kvsel_kv_compact: ";
  if (!kv || kv->num_kv_heads < 1 || !kv->k_pool || !kv->v_pool || kv->num_pages < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv descriptor with both pools is required");
  if (page_shift_of(kv->page_size) < 0 || kv->head_dim != kKcHD)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16, 32, 64, 128 or 256 are implemented");
  if (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pools must be 16-byte aligned");
  if (!block_table || !seq_lens || !keep || batch < 1 || max_pages < 1 || keep_stride < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "block_table, seq_lens, keep required; batch, max_pages, keep_stride >= 1");
  if ((scores || pos_map) && max_len < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "max_len >= 1 is required with scores or pos_map");
  if (!workspace || !aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "a 256-byte aligned workspace is required");
  const KcWs L = kc_ws_layout(batch, kv->num_kv_heads);
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(L.total));

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KcParams P;
  P.seq_lens = seq_lens;
  P.block_table = block_table;
  P.keep = keep;
  P.keep_count = keep_count;
  P.k_pool = static_cast<__nv_bfloat16*>(kv->k_pool);
  P.v_pool = static_cast<__nv_bfloat16*>(kv->v_pool);
  P.scores = scores;
  P.pos_map = pos_map;
  P.freed = freed_pages;
  P.n_keep = reinterpret_cast<int32_t*>(ws + L.n_off);
  P.first_move = reinterpret_cast<int32_t*>(ws + L.first_off);
  P.status = reinterpret_cast<int*>(ws);
  P.Hkv = kv->num_kv_heads;
  P.keep_stride = keep_stride;
  P.max_len = max_len;
  P.max_pages = max_pages;
  P.num_pages = kv->num_pages;
  P.page_shift = page_shift_of(kv->page_size);

  trace_before("kc_check", st);
  kc_check_kernel<<<batch, kKcCheckThreads, 0, st>>>(P);
  trace_after(st);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return cuda_fail(e, "kvsel_kv_compact (check launch)");

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  cfg.gridDim = dim3(kv->num_kv_heads, batch);
  cfg.blockDim = dim3(kKcThreads);
  cfg.dynamicSmemBytes = 0;
  trace_before("kc_move", st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kc_move_kernel, P);
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_kv_compact (move launch)");

  cfg.gridDim = dim3(batch);
  cfg.blockDim = dim3(kKcCheckThreads);
  cfg.dynamicSmemBytes = 0;
  trace_before("kc_truncate", st);
  e = cudaLaunchKernelEx(&cfg, kc_truncate_kernel, P);
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_kv_compact (truncate launch)");
  return KVSEL_OK;
}
