// Quest page selection for GQA decode (sm_103a).
//
// What it computes ("Long context, KV eviction and sparse attention", the
// sparse-selection section: Quest bounds a page's attention logit by the
// elementwise min and max of its keys and keeps the best pages).  For
// sequence b (S_b keys once the new token is appended) and q head h of kv
// head h / G:
//   bound[b, h, p] = sum_d max(q_d * kmin[p]_d, q_d * kmax[p]_d)   for every
//                    full page p < S_b / 16 (a Quest page is 16 tokens: one
//                    16-row tile of a pool page of 16 to 256 tokens)
//   pages[b, h]    = the budget_pages largest bounds, ties to the lower page
//                    (every full page when there are no more), ascending
//   o[b, h]        = softmax(scale * q . k) V over the tokens of pages[b, h]
//                    and of the trailing partial page, which is always kept
// Each q head chooses alone; the kv head streams the union of its heads'
// pages once and masks, per page, the heads that did not choose it.
//
// The bound uses max(q x, q y) = q+ y + q- x for x <= y (q+ = max(q, 0), q- =
// min(q, 0)): a plain dot product of bf16 values, run on the tensor cores.
//
// Kernels:
//   qu_meta_kernel   builds the per-page min / max of a prompt's keys: one
//                    warp per (page, kv head), a partial page over its valid
//                    tokens.  A page's pair sits beside its pool tile: pool
//                    page p, kv head h, tile j -> meta[p][h][j].
//   qu_bound_kernel  (page chunk, kv head, sequence), 8 warps: the CTA whose
//                    chunk holds the new token's page appends it (K and V
//                    rows, and the page's min / max) before its own bounds;
//                    then the bounds of 16 full pages x 8 heads (two such
//                    columns for 9..16 heads) per warp tile on the tensor cores (mma.sync: the pages' [min |
//                    max] rows, 512 bytes each, against the heads' [q- | q+],
//                    see below).
//   qu_topk_kernel   (q head, sequence): the top pages of the head's bounds
//                    (a register-resident radix select for rows of up to 16K
//                    pages, row_topk above), the kept pages marked in the kv
//                    head's page mask; the last of the G heads to finish
//                    lists the marked pages in ascending order with their
//                    pool tiles and head masks (the partial page last,
//                    for every head) and clears the mask.
//   qu_attn_kernel   (split, kv head, sequence), 4 warps: one 16-key tile per
//                    listed page (cp.async gather of its K and V rows into the
//                    swizzled tile, three stages per warp: two pages in
//                    flight while one is computed), attend_tile (9..16
//                    heads: attend_tile_wide) with the page's head mask; the last split of a (sequence, kv
//                    head) merges the splits into O and the last kv head
//                    publishes the length.
#include "attn_tile.cuh"
#include "row_topk.cuh"

namespace kvsel {

constexpr int kQuD = 128;
constexpr int kQuPage = 16;  // tokens per Quest page: one 16-row tile of a pool page of 16..256 tokens
constexpr int kQuMaxG = 16;  // q heads per kv head (bounds: one or two 8-head MMA columns)
constexpr int kQuBoundThreads = 256;
constexpr int kQuBoundPagesPerCta = 256;
constexpr int kQuTopkGroups = 8;          // row_topk (rows above 16K pages): up to 32K in registers
constexpr int kQuAttnWarps = 4;
constexpr int kQuAttnStages = 3;          // per warp
// the warps' merge scratch reuses the ring once every warp is done with it
constexpr size_t kQuAttnSmem = size_t(kQuAttnWarps) * kQuAttnStages * 8192 + 1024;
static_assert(size_t(kQuAttnWarps) * kTileMaxG * (kTileD + 2) * 4 <= size_t(kQuAttnWarps) * kQuAttnStages * 8192,
              "merge scratch fits in the ring");

struct QuParams {
  const int32_t* block_table;    // [B][max_pages]
  int32_t* seq_lens;             // [B]
  const __nv_bfloat16* q;        // [B][Hq][128]
  const __nv_bfloat16* k_new;    // [B][Hkv][128] or null
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  __nv_bfloat16* meta;           // [num_pages][Hkv][pool page / 16][2][128]: min row, max row
  float* bounds;                 // [B][Hq][max_qp]
  int32_t* sel;                  // [B][Hq][budget]
  uint32_t* mask;                // [B][Hkv][max_qp]: heads that chose each page (zero between calls)
  int32_t* ulist;                // [B][Hkv][max_qp]: listed pages, ascending
  int32_t* uphys;                // [B][Hkv][max_qp]: their pool tiles (qu_tile)
  uint32_t* umask;               // [B][Hkv][max_qp]: their head masks
  int32_t* ucount;               // [B][Hkv]
  unsigned* topk_cnt;            // [B][Hkv]: heads done (the last one lists)
  unsigned* merge_cnt;           // [B][Hkv]: splits done (the last one merges)
  unsigned* seq_cnt;             // [B]: kv heads merged (the last one publishes the length)
  float* part;                   // [B][Hkv][splits][kPartFloats]
  void* out;
  int* status;
  int B, max_pages, Hq, Hkv, G, num_pages, budget, chunks, splits, appended, out_f32;
  int page_shift;                // log2(pool page / 16)
  int max_qp;                    // Quest pages per block-table row: max_pages << page_shift
  float scale_log2;
};

__device__ __forceinline__ bool qu_len_ok(const QuParams& P, int b, int& S) {
  S = P.seq_lens[b] + P.appended;
  return S >= 0 && (S + kQuPage - 1) / kQuPage <= P.max_qp;
}

// Pool tile of Quest page t of sequence b, kv head kvh: the 16 rows from row
// 16 * tile of the pool and the min / max pair at meta + tile * 256.  A bad
// block-table entry is reported and read as page 0.
__device__ __forceinline__ int qu_tile_of(const int32_t* block_table, int max_pages, int num_pages, int Hkv,
                                          int page_shift, int* status, int b, int kvh, int t) {
  int phys = block_table[size_t(b) * max_pages + (t >> page_shift)];
  if (unsigned(phys) >= unsigned(num_pages)) {
    report(status, KVSEL_ERR_BAD_INDEX);
    phys = 0;
  }
  return ((phys * Hkv + kvh) << page_shift) | (t & ((1 << page_shift) - 1));
}
__device__ __forceinline__ int qu_tile(const QuParams& P, int b, int kvh, int t) {
  return qu_tile_of(P.block_table, P.max_pages, P.num_pages, P.Hkv, P.page_shift, P.status, b, kvh, t);
}

__device__ __forceinline__ void qu_cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ float bf16_at(uint4 v, int i) {
  const uint32_t w = (&v.x)[i >> 1];
  return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// ---------------------------------------------------------------------------
// Page min / max of a prompt: grid (ceil(max_qp / 4), Hkv, B), 4 warps, one
// Quest page each; lane l owns dimensions 4l .. 4l + 3.
struct QuMetaParams {
  const int32_t* block_table;
  const int32_t* seq_lens;
  const __nv_bfloat16* k_pool;
  __nv_bfloat16* meta;
  int* status;
  int max_pages, Hkv, num_pages, page_shift, max_qp;
};
__global__ void __launch_bounds__(128) qu_meta_kernel(const QuMetaParams P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int page = blockIdx.x * 4 + warp, kvh = blockIdx.y, b = blockIdx.z;
  const int S = P.seq_lens[b];
  if (S < 0 || (S + kQuPage - 1) / kQuPage > P.max_qp) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  if (page * kQuPage >= S) return;
  const int n = min(kQuPage, S - page * kQuPage);
  if (unsigned(P.block_table[size_t(b) * P.max_pages + (page >> P.page_shift)]) >= unsigned(P.num_pages)) {
    if (lane == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  const int tile = qu_tile_of(P.block_table, P.max_pages, P.num_pages, P.Hkv, P.page_shift, P.status, b, kvh, page);
  const __nv_bfloat16* rows = P.k_pool + size_t(tile) * kQuPage * kQuD;
  float mn[4], mx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mn[i] = INFINITY;
    mx[i] = -INFINITY;
  }
  for (int r = 0; r < n; ++r) {
    const uint2 v = *reinterpret_cast<const uint2*>(rows + size_t(r) * kQuD + 4 * lane);
    const uint4 w = make_uint4(v.x, v.y, 0u, 0u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float x = bf16_at(w, i);
      mn[i] = fminf(mn[i], x);
      mx[i] = fmaxf(mx[i], x);
    }
  }
  // min / max of bf16 values are bf16 values: the conversion back is exact
  __nv_bfloat16* m = P.meta + size_t(tile) * 2 * kQuD;
  *reinterpret_cast<uint2*>(m + 4 * lane) = make_uint2(pack_bf16x2(mn[0], mn[1]), pack_bf16x2(mn[2], mn[3]));
  *reinterpret_cast<uint2*>(m + kQuD + 4 * lane) =
      make_uint2(pack_bf16x2(mx[0], mx[1]), pack_bf16x2(mx[2], mx[3]));
}

// ---------------------------------------------------------------------------
// kWide: 9..16 q heads per kv head, heads 8.. in a second N = 8 column of MMAs
template <bool kWide>
__global__ void __launch_bounds__(kQuBoundThreads) qu_bound_kernel(const QuParams P) {
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  int S;
  if (!qu_len_ok(P, b, S)) {
    if (chunk == 0 && kvh == 0 && tid == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  const int npg = (S + kQuPage - 1) / kQuPage, n_full = S / kQuPage;
  const int p0 = int((long long)chunk * npg / P.chunks), p1 = int((long long)(chunk + 1) * npg / P.chunks);
  const int G = P.G;
  const int S_old = S - P.appended;
  const int pa = S_old / kQuPage;
  if (P.appended && pa >= p0 && pa < p1) {
    // the new token: K and V rows, then the page's min / max (first token: itself)
    const int tile = qu_tile(P, b, kvh, pa);
    const size_t row = size_t(tile) * kQuPage + (S_old % kQuPage);
    const __nv_bfloat16* kn = P.k_new + (size_t(b) * P.Hkv + kvh) * kQuD;
    const __nv_bfloat16* vn = P.v_new + (size_t(b) * P.Hkv + kvh) * kQuD;
    if (tid < 16) reinterpret_cast<uint4*>(P.k_pool + row * kQuD)[tid] = reinterpret_cast<const uint4*>(kn)[tid];
    else if (tid < 32) reinterpret_cast<uint4*>(P.v_pool + row * kQuD)[tid - 16] = reinterpret_cast<const uint4*>(vn)[tid - 16];
    else if (tid < 48) {
      const int u = tid - 32;  // 8 dimensions
      __nv_bfloat16* m = P.meta + size_t(tile) * 2 * kQuD;
      const uint4 x = reinterpret_cast<const uint4*>(kn)[u];
      uint4 lo = x, hi = x;
      if (S_old % kQuPage != 0) {
        const uint4 a = __ldcg(reinterpret_cast<const uint4*>(m) + u);
        const uint4 c = __ldcg(reinterpret_cast<const uint4*>(m + kQuD) + u);
        uint32_t* lw = &lo.x;
        uint32_t* hw = &hi.x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          lw[i] = pack_bf16x2(fminf(bf16_at(a, 2 * i), bf16_at(x, 2 * i)), fminf(bf16_at(a, 2 * i + 1), bf16_at(x, 2 * i + 1)));
          hw[i] = pack_bf16x2(fmaxf(bf16_at(c, 2 * i), bf16_at(x, 2 * i)), fmaxf(bf16_at(c, 2 * i + 1), bf16_at(x, 2 * i + 1)));
        }
      }
      reinterpret_cast<uint4*>(m)[u] = lo;
      reinterpret_cast<uint4*>(m + kQuD)[u] = hi;
    }
  }
  // Bounds on the tensor cores: with x <= y, max(q x, q y) = q+ y + q- x (q+ = max(q, 0),
  // q- = min(q, 0)), so bound[p][h] = sum over the 256 entries of page p's [min | max]
  // row times head h's [q- | q+]: an M = 16 pages x N = 8 heads x K = 256 product per
  // tile, every operand an exact bf16 value.  K is permuted so that each lane reads
  // 16-byte runs: for 16-byte unit u (physical entries 32u + 8c .. + 7, c = lane % 4)
  // k-step 2u + v takes entries 32u + 8c + 4v + {0, 1} as logical k {2c, 2c + 1} and
  // + {2, 3} as {2c + 8, 2c + 9}, on A and B alike.
  const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, cq = lane & 3;
  constexpr int kCols = kWide ? 2 : 1;  // 8-head columns: heads 8 j .. 8 j + 7
  uint32_t bfr[kCols][16][2];
#pragma unroll
  for (int j = 0; j < kCols; ++j) {
    const int hq = 8 * j + gq;
    uint4 qraw[4] = {};
    if (hq < G) {
      const uint4* qrow = reinterpret_cast<const uint4*>(P.q + (size_t(b) * P.Hq + size_t(kvh) * G + hq) * kQuD);
#pragma unroll
      for (int u = 0; u < 4; ++u) qraw[u] = qrow[4 * u + cq];  // dims 32u + 8c .. + 7
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 x = qraw[u & 3];
      const bool plus = u >= 4;  // entries 128.. multiply the max row
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t v = (&x.x)[i];
        uint32_t r = 0u;
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          const uint32_t e = (v >> (16 * hlf)) & 0xFFFFu;
          const bool neg = (e & 0x8000u) != 0u;
          r |= ((plus ? !neg : neg) ? e : 0u) << (16 * hlf);
        }
        w[i] = r;
      }
      bfr[j][2 * u][0] = w[0];
      bfr[j][2 * u][1] = w[1];
      bfr[j][2 * u + 1][0] = w[2];
      bfr[j][2 * u + 1][1] = w[3];
    }
  }
  __syncthreads();  // orders the append's min / max before the reads below
  const int pe = min(p1, n_full);
  float* bnd = P.bounds + (size_t(b) * P.Hq + size_t(kvh) * G) * P.max_qp;
  constexpr int kWarps = kQuBoundThreads / 32;
#pragma unroll 1
  for (int tp = p0 + warp * 16; tp < pe; tp += kWarps * 16) {
    const int pg0 = tp + gq, pg1 = tp + gq + 8;
    const uint4* r0 = pg0 < pe ? reinterpret_cast<const uint4*>(P.meta + size_t(qu_tile(P, b, kvh, pg0)) * 2 * kQuD) : nullptr;
    const uint4* r1 = pg1 < pe ? reinterpret_cast<const uint4*>(P.meta + size_t(qu_tile(P, b, kvh, pg1)) * 2 * kQuD) : nullptr;
    uint4 x0[8], x1[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      x0[u] = r0 ? __ldcg(r0 + 4 * u + cq) : make_uint4(0u, 0u, 0u, 0u);
      x1[u] = r1 ? __ldcg(r1 + 4 * u + cq) : make_uint4(0u, 0u, 0u, 0u);
    }
    float c[kCols][4] = {};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        mma_bf16_16816(c[j], x0[u].x, x1[u].x, x0[u].y, x1[u].y, bfr[j][2 * u][0], bfr[j][2 * u][1]);
        mma_bf16_16816(c[j], x0[u].z, x1[u].z, x0[u].w, x1[u].w, bfr[j][2 * u + 1][0], bfr[j][2 * u + 1][1]);
      }
    }
    // c[j]: pages (gq, gq + 8) x heads (8 j + 2 cq, 8 j + 2 cq + 1)
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int h0 = 8 * j + 2 * cq, h1 = h0 + 1;
      if (pg0 < pe) {
        if (h0 < G) bnd[size_t(h0) * P.max_qp + pg0] = c[j][0];
        if (h1 < G) bnd[size_t(h1) * P.max_qp + pg0] = c[j][1];
      }
      if (pg1 < pe) {
        if (h0 < G) bnd[size_t(h0) * P.max_qp + pg1] = c[j][2];
        if (h1 < G) bnd[size_t(h1) * P.max_qp + pg1] = c[j][3];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Top-k of a row of up to kQuSmallRow fp32 bounds by one 1024-thread CTA
// (k < n): thread t holds positions 16t .. 16t + 15 as order keys in
// registers; a radix select finds the k-th key T (four 8-bit digits, most
// significant first; the histogram adds are aggregated per warp with
// match_any, since the bounds' leading bits are nearly all alike), then an
// ordered emission keeps every key above T and the first `remaining` equal to
// it (ties to the lower position), in ascending position order.
constexpr int kQuSmallPer = 16;
constexpr int kQuSmallRow = kRkThreads * kQuSmallPer;
template <class Emit>
__device__ __forceinline__ void qu_small_topk(const float* row, int n, int k, uint32_t* hist, uint32_t* tmp,
                                              uint32_t* bc, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t kk[kQuSmallPer];
  const int p0 = tid * kQuSmallPer;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && p0 + kQuSmallPer <= n) {
#pragma unroll
    for (int j = 0; j < kQuSmallPer; j += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(row + p0 + j));
      kk[j] = order_key(v.x);
      kk[j + 1] = order_key(v.y);
      kk[j + 2] = order_key(v.z);
      kk[j + 3] = order_key(v.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kQuSmallPer; ++j) kk[j] = p0 + j < n ? order_key(__ldcg(row + p0 + j)) : 0u;
  }
  uint32_t prefix = 0u, mask = 0u, remaining = uint32_t(k);
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kRkThreads) hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kQuSmallPer; ++j) {
      const bool live = p0 + j < n && (kk[j] & mask) == prefix;
      const uint32_t d = live ? (kk[j] >> shift) & 255u : 256u;  // 256: not counted
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (live && (peers & rk_lanemask_lt()) == 0u) atomicAdd(hist + d, uint32_t(__popc(peers)));
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
      const uint32_t above = incl - tot;
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
  const uint32_t T = prefix;
  uint32_t neq = 0u;
#pragma unroll
  for (int j = 0; j < kQuSmallPer; ++j) neq += (p0 + j < n && kk[j] == T) ? 1u : 0u;
  uint32_t tot;
  uint32_t eq_rank = rk_block_excl_scan(neq, tmp, tot);
  uint32_t ntake = 0u;
  uint32_t take = 0u;  // bit j: position p0 + j is kept
#pragma unroll
  for (int j = 0; j < kQuSmallPer; ++j) {
    bool t = false;
    if (p0 + j < n) {
      if (kk[j] > T) t = true;
      else if (kk[j] == T) t = eq_rank++ < remaining;
    }
    take |= (t ? 1u : 0u) << j;
    ntake += t ? 1u : 0u;
  }
  uint32_t o = rk_block_excl_scan(ntake, tmp, tot);
#pragma unroll
  for (int j = 0; j < kQuSmallPer; ++j)
    if ((take >> j) & 1u) emit(int(o++), p0 + j);
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRkThreads) qu_topk_kernel(const QuParams P) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  RowTopkSmem& sm = *reinterpret_cast<RowTopkSmem*>(tk_smem);
  __shared__ int s_last;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int G = P.G, kvh = h / G, g = h % G;
  int S;
  if (!qu_len_ok(P, b, S)) return;
  const int n_full = S / kQuPage, k = P.budget;
  int32_t* sel = P.sel + (size_t(b) * P.Hq + h) * k;
  uint32_t* msk = P.mask + (size_t(b) * P.Hkv + kvh) * P.max_qp;
  const uint32_t bit = 1u << g;
  if (n_full <= k) {
    for (int i = tid; i < k; i += kRkThreads) {
      sel[i] = i < n_full ? i : -1;
      if (i < n_full) atomicOr(msk + i, bit);
    }
  } else if (n_full <= kQuSmallRow) {
    const float* row = P.bounds + (size_t(b) * P.Hq + h) * P.max_qp;
    qu_small_topk(row, n_full, k, sm.hist, sm.wtot[0], sm.wtot[1], [&](int i, int p) {
      sel[i] = p;
      atomicOr(msk + p, bit);
    });
  } else {
    const float* row = P.bounds + (size_t(b) * P.Hq + h) * P.max_qp;
    const F32RowKeys src{row, 0, n_full, (reinterpret_cast<uintptr_t>(row) & 15u) == 0};
    row_topk<kQuTopkGroups>(src, k, 0u, sm, [&](int i, int p) {
      sel[i] = p;
      atomicOr(msk + p, bit);
    });
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    unsigned* cnt = P.topk_cnt + size_t(b) * P.Hkv + kvh;
    s_last = atomicAdd(cnt, 1u) + 1u == unsigned(G);
    if (s_last) {
      *cnt = 0u;  // every head has arrived: ready for the next call
      __threadfence();
    }
  }
  __syncthreads();
  if (!s_last) return;
  // list the marked pages in ascending order (block scan per round of 1024)
  int32_t* ul = P.ulist + (size_t(b) * P.Hkv + kvh) * P.max_qp;
  int32_t* uph = P.uphys + (size_t(b) * P.Hkv + kvh) * P.max_qp;
  uint32_t* um = P.umask + (size_t(b) * P.Hkv + kvh) * P.max_qp;
  uint32_t total_all = 0;
  for (int r0 = 0; r0 < n_full; r0 += kRkThreads) {
    const int i = r0 + tid;
    const uint32_t m = i < n_full ? __ldcg(msk + i) : 0u;
    uint32_t tot;
    const uint32_t off = rk_block_excl_scan(m != 0u ? 1u : 0u, sm.wtot[0], tot);
    if (m != 0u) {
      ul[total_all + off] = i;
      uph[total_all + off] = qu_tile(P, b, kvh, i);
      um[total_all + off] = m;
      msk[i] = 0u;
    }
    total_all += tot;
  }
  if (tid == 0) {
    int n = int(total_all);
    if (S % kQuPage != 0) {  // the partial page, for every head
      ul[n] = n_full;
      uph[n] = qu_tile(P, b, kvh, n_full);
      um[n] = (G >= 32) ? 0xFFFFFFFFu : ((1u << G) - 1u);
      ++n;
    }
    P.ucount[size_t(b) * P.Hkv + kvh] = n;
  }
}

// ---------------------------------------------------------------------------
// kWide: 9..16 q heads per kv head (attend_tile_wide: head g + 8 in MMA rows 8..15)
template <bool kWide>
__global__ void __launch_bounds__(kQuAttnWarps * 32) qu_attn_kernel(const QuParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* wo = reinterpret_cast<float*>(smem);  // after the page loop
  __shared__ int s_last;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int S;
  if (!qu_len_ok(P, b, S)) return;
  const int n = P.ucount[size_t(b) * P.Hkv + kvh];
  const int n_full = S / kQuPage, tail = S % kQuPage;
  const int t0 = int((long long)split * n / P.splits), t1 = int((long long)(split + 1) * n / P.splits);
  const int G = P.G, g = lane >> 2, qd = lane & 3;
  const bool head_ok = g < G, head_ok2 = kWide && g + 8 < G;
  const size_t lbase = (size_t(b) * P.Hkv + kvh) * P.max_qp;
  const uint32_t wbuf = smem_u32(smem + warp * kQuAttnStages * 8192);
  const int num_tiles = (P.num_pages * P.Hkv) << P.page_shift;

  uint32_t qa[8][2], qb[8][2];
  load_q_frags(P.q + (size_t(b) * P.Hq + kvh * G + (head_ok ? g : 0)) * kQuD, head_ok, qd, qa);
  if (kWide) load_q_frags(P.q + (size_t(b) * P.Hq + kvh * G + (head_ok2 ? g + 8 : 0)) * kQuD, head_ok2, qd, qb);
  TileState st;
  st.init();

  // this warp's list entries are t0 + warp + 4 i; lane j holds entry cbase + j of
  // the current chunk of 32 (page, pool tile, head mask), read ahead in one go
  const int nw = t0 + warp < t1 ? (t1 - t0 - warp + kQuAttnWarps - 1) / kQuAttnWarps : 0;
  int cbase = 0, c_page = 0, c_tile = 0;
  uint32_t c_mask = 0u;
  auto load_chunk = [&](int base) {
    const int e = t0 + warp + kQuAttnWarps * (base + lane);
    const bool ok = base + lane < nw;
    c_page = ok ? P.ulist[lbase + e] : 0;
    c_tile = ok ? P.uphys[lbase + e] : 0;
    c_mask = ok ? P.umask[lbase + e] : 0u;
  };
  auto entry = [&](int i, int& page, int& tile, uint32_t& m) {  // called by the whole warp
    if (i - cbase < 32) {
      page = __shfl_sync(0xffffffffu, c_page, i - cbase);
      tile = __shfl_sync(0xffffffffu, c_tile, i - cbase);
      m = __shfl_sync(0xffffffffu, c_mask, i - cbase);
    } else {  // read-ahead past the chunk: straight from the list
      const size_t e = lbase + t0 + warp + size_t(kQuAttnWarps) * i;
      page = P.ulist[e];
      tile = P.uphys[e];
      m = P.umask[e];
    }
  };
  load_chunk(0);

  // entry i into stage s: its page's 16 K rows then 16 V rows (rows past a
  // partial page's tokens are zero-filled)
  auto gather = [&](int i, int s) {
    int page, tile;
    uint32_t m;
    entry(i, page, tile, m);
    if (unsigned(tile) >= unsigned(num_tiles)) tile = 0;  // a bad entry was reported when the list was built
    const int valid = page == n_full ? tail : kQuPage;
    const size_t base = size_t(tile) * kQuPage * kQuD;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int c = lane + 32 * k;
      const int row = c >> 4, u = c & 15;
      const int r16 = row & 15;
      const __nv_bfloat16* src = (row < 16 ? P.k_pool : P.v_pool) + base + size_t(r16) * kQuD + u * 8;
      qu_cp_async16(wbuf + s * 8192 + (row < 16 ? 0 : 4096) + tile_unit_off(r16, u), src, r16 < valid);
    }
  };
  auto commit = []() { asm volatile("cp.async.commit_group;" ::: "memory"); };

  // every iteration commits one group (empty past the end), so the current
  // entry's group is always the third most recent
#pragma unroll
  for (int k = 0; k < kQuAttnStages - 1; ++k) {
    if (k < nw) gather(k, k);
    commit();
  }
  int s = 0;
#pragma unroll 1
  for (int i = 0; i < nw; ++i) {
    if (i - cbase == 32) {  // the chunk is used up (the read-ahead went straight to the list)
      cbase += 32;
      load_chunk(cbase);
    }
    const int in = i + kQuAttnStages - 1;
    if (in < nw) gather(in, s == 0 ? kQuAttnStages - 1 : s - 1);
    commit();
    asm volatile("cp.async.wait_group %0;" ::"n"(kQuAttnStages - 1) : "memory");
    __syncwarp();
    int page, tile;
    uint32_t m;
    entry(i, page, tile, m);
    const bool on = head_ok && ((m >> g) & 1u);
    const int valid = page == n_full ? tail : kQuPage;
    if (kWide) {
      const bool on2 = head_ok2 && ((m >> (g + 8)) & 1u);
      attend_tile_wide(wbuf + s * 8192, wbuf + s * 8192 + 4096, qa, qb, valid, P.scale_log2, st, on, on2);
    } else {
      float x0, x1, x2, x3;
      attend_tile(wbuf + s * 8192, wbuf + s * 8192 + 4096, qa, valid, P.scale_log2, st, x0, x1, x2, x3, on);
    }
    __syncwarp();
    s = s + 1 == kQuAttnStages ? 0 : s + 1;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();  // every warp is done with the ring: it becomes the merge scratch
  float* slot = P.part + ((size_t(b) * P.Hkv + kvh) * P.splits + split) * kPartFloats;
  merge_warps_to_slot<kQuAttnWarps, kWide>(st, wo, slot, G);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    unsigned* cnt = P.merge_cnt + size_t(b) * P.Hkv + kvh;
    s_last = atomicAdd(cnt, 1u) + 1u == unsigned(P.splits);
    if (s_last) {
      *cnt = 0u;
      __threadfence();
    }
  }
  __syncthreads();
  if (s_last) {
    merge_split_slots(P.part + (size_t(b) * P.Hkv + kvh) * P.splits * kPartFloats, P.splits, G, P.out,
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
struct QuWs {
  size_t cnt, bounds, sel, mask, ulist, uphys, umask, ucount, part, total;
};
QuWs qu_ws_layout(int batch, int Hq, int Hkv, int max_qp, int budget, bool own_bounds, bool own_sel) {
  QuWs w;
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.cnt = take((size_t(batch) * Hkv * 2 + batch) * 4);
  w.bounds = own_bounds ? take(size_t(batch) * Hq * max_qp * 4) : 0;
  w.sel = own_sel ? take(size_t(batch) * Hq * budget * 4) : 0;
  w.mask = take(size_t(batch) * Hkv * max_qp * 4);
  w.ulist = take(size_t(batch) * Hkv * max_qp * 4);
  w.uphys = take(size_t(batch) * Hkv * max_qp * 4);
  w.umask = take(size_t(batch) * Hkv * max_qp * 4);
  w.ucount = take(size_t(batch) * Hkv * 4);
  w.part = take(size_t(batch) * Hkv * kTileMaxSplits * kPartFloats * 4);
  w.total = off;
  return w;
}
}  // namespace

extern "C" kvsel_status kvsel_quest_page_meta(const kvsel_paged_kv* kv, const int32_t* block_table, int max_pages,
                                              const int32_t* seq_lens, int batch, void* page_meta,
                                              void* status_word, void* stream) {
  const std::string fn = "kvsel_quest_page_meta: ";
  if (!kv || !kv->k_pool || !block_table || !seq_lens || !page_meta || !status_word || batch < 1 || max_pages < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "kv, block_table, seq_lens, page_meta, status_word required; "
                                            "batch, max_pages >= 1");
  if (kv->head_dim != kQuD || page_shift_of(kv->page_size) < 0)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "head_dim 128 and page_size 16, 32, 64, 128 or 256 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_pages < 1 || batch > 65535 || kv->num_kv_heads > 65535)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_kv_heads and num_pages >= 1; batch, num_kv_heads <= 65535");
  if ((long long)max_pages * kv->page_size >= (1LL << 31) ||
      (long long)kv->num_pages * kv->num_kv_heads * kv->page_size >= (1LL << 31))
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "max_pages * page_size and num_pages * num_kv_heads * page_size < 2^31");
  if (!aligned(kv->k_pool, 16) || !aligned(page_meta, 16) || !aligned(status_word, 4))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "K pool and page_meta must be 16-byte aligned");
  QuMetaParams P;
  P.block_table = block_table;
  P.seq_lens = seq_lens;
  P.k_pool = static_cast<const __nv_bfloat16*>(kv->k_pool);
  P.meta = static_cast<__nv_bfloat16*>(page_meta);
  P.status = static_cast<int*>(status_word);
  P.max_pages = max_pages;
  P.Hkv = kv->num_kv_heads;
  P.num_pages = kv->num_pages;
  P.page_shift = page_shift_of(kv->page_size);
  P.max_qp = max_pages << P.page_shift;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  trace_before("qu_meta", st);
  qu_meta_kernel<<<dim3((P.max_qp + 3) / 4, P.Hkv, batch), 128, 0, st>>>(P);
  const cudaError_t e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_quest_page_meta (launch)");
  return KVSEL_OK;
}

extern "C" size_t kvsel_quest_decode_workspace(const kvsel_paged_kv* kv, int batch, int max_pages, int budget_pages,
                                               int with_bounds_out, int with_pages_out) {
  if (!kv || batch < 1 || max_pages < 1 || budget_pages < 1 || kv->num_kv_heads < 1 ||
      kv->num_q_heads % kv->num_kv_heads != 0 || page_shift_of(kv->page_size) < 0 ||
      (long long)max_pages * kv->page_size >= (1LL << 31))
    return 0;
  return qu_ws_layout(batch, kv->num_q_heads, kv->num_kv_heads, max_pages << page_shift_of(kv->page_size),
                      budget_pages, with_bounds_out == 0, with_pages_out == 0).total;
}

extern "C" kvsel_status kvsel_quest_decode(const kvsel_paged_kv* kv, const int32_t* block_table, int max_pages,
                                           int32_t* seq_lens, int batch, const void* q, const void* k_new,
                                           const void* v_new, void* page_meta, int budget_pages, float scale,
                                           void* out, int out_dtype, int32_t* pages_out, float* bounds_out,
                                           void* workspace, size_t ws_bytes, void* stream) {
  const std::string fn = "kvsel_quest_decode: ";
  if (!kv || !kv->k_pool || !kv->v_pool) return fail(KVSEL_ERR_INVALID_ARG, fn + "kv pools must be non-NULL");
  if (kv->head_dim != kQuD || page_shift_of(kv->page_size) < 0)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "head_dim 128 and page_size 16, 32, 64, 128 or 256 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (G > kQuMaxG) return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 16 q heads per kv head");
  if (!block_table || !seq_lens || !q || !out || !page_meta || batch < 1 || max_pages < 1 || budget_pages < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "block_table, seq_lens, q, out, page_meta are required; batch, "
                                            "max_pages, budget_pages >= 1");
  if ((k_new == nullptr) != (v_new == nullptr))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "k_new and v_new must both be given or both NULL");
  if (out_dtype != KVSEL_BF16 && out_dtype != KVSEL_F32)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "out_dtype must be KVSEL_BF16 or KVSEL_F32");
  if (batch > 65535 || Hq > 65535 || (long long)max_pages * kv->page_size >= (1LL << 31) ||
      (long long)kv->num_pages * Hkv * kv->page_size >= (1LL << 31) || kv->num_pages < 1)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "batch, num_q_heads <= 65535; max_pages * page_size and num_pages * "
                                            "num_kv_heads * page_size < 2^31");
  if (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16) || !aligned(q, 16) || !aligned(page_meta, 16) ||
      (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pools, q, k_new, v_new and page_meta must be 16-byte aligned");
  const int page_shift = page_shift_of(kv->page_size);
  const int max_qp = max_pages << page_shift;  // Quest pages (16 tokens) per block-table row
  const QuWs L = qu_ws_layout(batch, Hq, Hkv, max_qp, budget_pages, bounds_out == nullptr, pages_out == nullptr);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace missing, misaligned or smaller than " +
                                           std::to_string(L.total));

  const int sms = sm_count();
  const int list_max = std::min(max_qp, G * budget_pages + 1);
  int splits = std::max(1, (sms * 2) / (batch * Hkv));  // one wave at two CTAs per SM
  splits = std::min(splits, std::max(1, (list_max + 7) / 8));
  splits = std::min(splits, kTileMaxSplits);
  const int chunks = std::max(1, std::min(65535, (max_qp + kQuBoundPagesPerCta - 1) / kQuBoundPagesPerCta));

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  QuParams P;
  P.block_table = block_table;
  P.seq_lens = seq_lens;
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.k_new = static_cast<const __nv_bfloat16*>(k_new);
  P.v_new = static_cast<const __nv_bfloat16*>(v_new);
  P.k_pool = static_cast<__nv_bfloat16*>(kv->k_pool);
  P.v_pool = static_cast<__nv_bfloat16*>(kv->v_pool);
  P.meta = static_cast<__nv_bfloat16*>(page_meta);
  P.bounds = bounds_out ? bounds_out : reinterpret_cast<float*>(ws + L.bounds);
  P.sel = pages_out ? pages_out : reinterpret_cast<int32_t*>(ws + L.sel);
  P.mask = reinterpret_cast<uint32_t*>(ws + L.mask);
  P.ulist = reinterpret_cast<int32_t*>(ws + L.ulist);
  P.uphys = reinterpret_cast<int32_t*>(ws + L.uphys);
  P.umask = reinterpret_cast<uint32_t*>(ws + L.umask);
  P.ucount = reinterpret_cast<int32_t*>(ws + L.ucount);
  P.topk_cnt = reinterpret_cast<unsigned*>(ws + L.cnt);
  P.merge_cnt = P.topk_cnt + size_t(batch) * Hkv;
  P.seq_cnt = P.merge_cnt + size_t(batch) * Hkv;
  P.part = reinterpret_cast<float*>(ws + L.part);
  P.out = out;
  P.status = reinterpret_cast<int*>(ws);
  P.B = batch;
  P.max_pages = max_pages;
  P.page_shift = page_shift;
  P.max_qp = max_qp;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.num_pages = kv->num_pages;
  P.budget = budget_pages;
  P.chunks = chunks;
  P.splits = splits;
  P.appended = k_new ? 1 : 0;
  P.out_f32 = out_dtype == KVSEL_F32;
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    cudaError_t e0 = smem_limit_once(reinterpret_cast<const void*>(qu_attn_kernel<false>), int(kQuAttnSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(qu_attn_kernel<true>), int(kQuAttnSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(qu_topk_kernel), int(sizeof(RowTopkSmem)));
    if (e0 != cudaSuccess) return cuda_fail(e0, "kvsel_quest_decode (attribute)");
  }
  cudaError_t e;
#define KVSEL_QU_LAUNCH(name, kernel, grid, block, smem)                 \
  trace_before(name, st);                                                \
  kernel<<<grid, block, smem, st>>>(P);                                  \
  e = cudaGetLastError();                                                \
  trace_after(st);                                                       \
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_quest_decode (" name ")");
  if (G > 8) {
    KVSEL_QU_LAUNCH("qu_bound", qu_bound_kernel<true>, dim3(chunks, Hkv, batch), kQuBoundThreads, 0)
  } else {
    KVSEL_QU_LAUNCH("qu_bound", qu_bound_kernel<false>, dim3(chunks, Hkv, batch), kQuBoundThreads, 0)
  }
  KVSEL_QU_LAUNCH("qu_topk", qu_topk_kernel, dim3(Hq, batch), kRkThreads, sizeof(RowTopkSmem))
  if (G > 8) {
    KVSEL_QU_LAUNCH("qu_attn", qu_attn_kernel<true>, dim3(splits, Hkv, batch), kQuAttnWarps * 32, kQuAttnSmem)
  } else {
    KVSEL_QU_LAUNCH("qu_attn", qu_attn_kernel<false>, dim3(splits, Hkv, batch), kQuAttnWarps * 32, kQuAttnSmem)
  }
#undef KVSEL_QU_LAUNCH
  return KVSEL_OK;
}
