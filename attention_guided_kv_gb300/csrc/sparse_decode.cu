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
// Kernels (three launches on the caller's stream, chained by programmatic
// launch so each one's launch overlaps its predecessor's tail):
//   sd_index_kernel   (CTA range of 16-token tiles, sequence): streams the
//                     sequence's indexer keys with 16-byte loads, four tiles
//                     in flight per warp; the dot products run on mma.sync
//                     (16 tokens x 16 dims x 8 heads per MMA, the dims
//                     permuted per lane so that a lane's 16-byte run of a key
//                     row feeds two k-steps); writes the scores and adds their
//                     top 12 key bits to a per-row histogram (a shared-memory
//                     histogram per CTA, flushed once); also writes the
//                     appended token's K, V and indexer key.
//   sd_select_cluster_kernel  (8 CTAs, sequence), one 8-CTA cluster of 1024
//                     threads per row, rows up to 256K positions: each CTA
//                     holds a chunk of the row's scores in shared memory,
//                     takes the k-th key's top 12 bits from the histogram,
//                     compacts its candidates (keys in or above that bin) in
//                     one sweep, and resolves the other 20 bits in two radix
//                     passes whose counts the cluster sums through
//                     distributed shared memory; every CTA then writes its
//                     own kept positions, in ascending order, at offsets
//                     from the cluster's kept counts.
//   sd_select_kernel  (slices, sequence), longer rows, 1024 threads: every CTA finds, from
//                     the histogram, the bin holding the k-th largest score
//                     and appends the positions of its slice scoring in or
//                     above that bin to a candidate list (a few thousand at
//                     the 128K shape); the last CTA of the row selects the
//                     exact top_k among the candidates (radix select on the
//                     keys, bitmaps over the positions for the tie rule and
//                     the ascending order), resolves each selected position's
//                     page, and resets the row's histogram and counters.
//                     Lists too long for shared memory fall back to the
//                     whole-row select (row_topk) in the same CTA.
//   sd_attn_kernel    (splits, kv head, sequence), the splits of a (sequence,
//                     kv head) one thread-block cluster: each warp gathers 16
//                     selected rows of K and V at a time with cp.async into
//                     the swizzled tile layout (three tiles in flight; the
//                     pool rows, resolved by the select, loaded four tiles at
//                     a time and shared by shuffles) and runs the shared
//                     mma.sync tile; the 4 warps merge per CTA into shared
//                     memory, the cluster's CTAs merge the splits through
//                     distributed shared memory (each writes a slice of O),
//                     and the last kv head of a sequence publishes its length
#include "attn_tile.cuh"
#include "row_topk.cuh"

namespace kvsel {

constexpr int kSdD = 128;
constexpr int kSdPage = 16;  // the smallest page; pools may use 16 << page_shift tokens per page
constexpr int kSdDi = 64;
constexpr int kSdMaxHi = 8;
constexpr int kSdTopkGroups = 8;         // whole-row fallback: rows up to 32K stay in registers
constexpr int kSdMaxLen = 1 << 28;
constexpr int kSdMaxG = kTileMaxG;
constexpr int kSdPartFloats = kPartFloats;
constexpr int kSdAttnWarps = 4;
constexpr int kSdAttnStages = 3;         // gathered tiles in flight per warp
constexpr int kSdMaxClusterSplits = 8;   // splits of a (sequence, kv head): one portable cluster
// the warps' rings; the CTA's merge scratch reuses them once every tile is consumed
constexpr size_t kSdAttnRing = size_t(kSdAttnWarps) * kSdAttnStages * 8192;
static_assert(kSdAttnRing >= size_t(kSdAttnWarps) * kSdMaxG * (kSdD + 2) * 4, "merge scratch fits in the rings");
constexpr size_t kSdAttnSmem = kSdAttnRing + 1024;
constexpr int kSdIdxWarps = 8;           // indexer CTA: 8 warps
constexpr int kSdIdxRing = 4;            // tiles of 16 keys in a warp's copy ring (3 in flight)
constexpr int kSdIdxTileBytes = 16 * 128; // 16 keys x 64 bf16
constexpr size_t kSdIdxSmem = size_t(1 << 12) * 4 + size_t(kSdIdxWarps) * kSdIdxRing * kSdIdxTileBytes;
constexpr int kSdHistBits = 12;          // histogram of the top 12 bits of a score's order key
constexpr int kSdHistBins = 1 << kSdHistBits;
constexpr int kSdSelThreads = 1024;
constexpr int kSdCandCap = 12288;        // candidates per row the final select holds (12 per thread): a
                                         // row whose scores are all <= 0 ties thousands of keys at 0
constexpr int kSdSelSlice = 16 * kSdSelThreads;  // positions a select CTA scans (16 per thread)
constexpr int kSdSliceCap = 2048;        // candidates a slice may hand over (more: whole-row select)
constexpr int kSdMaxSlices = kSdSelThreads;  // slices the final select reads in one pass (rows to 16M)

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
  uint32_t* hist;                  // [B][kSdHistBins]: score counts by top key bits (zero between calls)
  uint32_t* subhist;               // [B][kSdHistBins]: the threshold bin's counts by the next 12 bits (zero)
  unsigned* cand_cnt;              // [B][slices]: candidates each select slice found
  unsigned* row_done;              // [B]: select CTAs finished (zero between calls)
  uint32_t* cand_key;              // [B][slices][kSdSliceCap], each slice in position order
  int32_t* cand_pos;               // [B][slices][kSdSliceCap]
  int32_t* cand_row;               // [B][slices][kSdSliceCap]: the candidate's pool row for kv head 0
  int32_t* sel;                    // [B][top_k]
  int32_t* sel_row;                // [B][top_k]: pool row of each selected position for kv head 0
  unsigned* seq_cnt;               // [B]: kv heads merged (the last one publishes the length)
  int32_t* nsel;                   // [B]
  int32_t* topk_out;               // [B][top_k] or null
  void* out;
  int* status;
  int B, max_pages, Hq, Hkv, G, Hi, num_pages, max_len, top_k, idx_ctas, slices, splits, appended, out_f32;
  int scores_vec;                  // score rows are 16-byte aligned (float4 reads)
  int page_shift;                  // log2(page_size / 16)
  float scale_log2;
};

__device__ __forceinline__ bool sd_len_ok(const SdParams& P, int b, int& S) {
  S = P.seq_lens[b] + P.appended;
  return S >= 0 && S <= P.max_len && (((long long)S + (kSdPage << P.page_shift) - 1) >> (4 + P.page_shift)) <= P.max_pages;
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
// Indexer.  Lane (g, q) of a warp holds, for a tile of 16 tokens, rows g and
// g + 8 as two 16-byte runs each: dims 8q..8q+7 and 32+8q..32+8q+7.  MMA
// k-step t takes the half (t & 1) of run (t >> 1) as its logical k's
// {2q, 2q+1 | 2q+8, 2q+9}; the indexer query (the B operand) is read with the
// same permutation, so each product pairs the same physical dims.
// One warp's copy of a 16-key tile (16 rows of 128 B) into a ring slot, 16-byte chunk c of row r
// stored at chunk c ^ (r & 7), so that the fragment reads below hit eight different bank groups;
// rows at or past the length are zero-filled.
__device__ __forceinline__ void sd_idx_tile_copy(uint32_t slot, const __nv_bfloat16* tile, int rows, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = lane + 32 * i, r = q >> 3, ch = q & 7;
    const bool ok = r < rows;
    cp_async16(slot + r * 128 + ((ch ^ (r & 7)) << 4), tile + (ok ? r * kSdDi + ch * 8 : 0), ok);
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__global__ void __launch_bounds__(kSdIdxWarps * 32) sd_index_kernel(const SdParams P) {
  extern __shared__ __align__(128) uint8_t idx_smem[];
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(idx_smem);  // [kSdHistBins]
  // launched early when the previous kernel allows it (the previous step's attention does, once its
  // gathers are done): nothing is read or written before that kernel has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the select waits for this grid
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int S;
  if (!sd_len_ok(P, b, S)) {
    if (c == 0 && tid == 0) report(P.status, KVSEL_ERR_BAD_INDEX);
    return;
  }
  const int S_old = S - P.appended;
  const int tiles = (S + 15) / 16;
  const int t0 = int((long long)tiles * c / P.idx_ctas), t1 = int((long long)tiles * (c + 1) / P.idx_ctas);
  if (P.appended && S_old / 16 >= t0 && S_old / 16 < t1) {
    // this CTA covers the appended token: its K, V (every kv head) and indexer key (which this
    // CTA's own copies below read back from L2)
    const int phys = P.block_table[size_t(b) * P.max_pages + (S_old >> (4 + P.page_shift))];
    if (unsigned(phys) < unsigned(P.num_pages)) {
      for (int i = tid; i < P.Hkv * 32; i += blockDim.x) {
        const int kvh = i >> 5, t = i & 15;
        const bool isv = (i & 31) >= 16;
        const size_t row = ((size_t(phys) * P.Hkv + kvh) << (4 + P.page_shift)) +
                           (S_old & ((kSdPage << P.page_shift) - 1));
        const uint4* src = reinterpret_cast<const uint4*>((isv ? P.v_new : P.k_new) +
                                                          (size_t(b) * P.Hkv + kvh) * kSdD);
        reinterpret_cast<uint4*>((isv ? P.v_pool : P.k_pool) + row * kSdD)[t] = src[t];
      }
    } else if (tid == 0) {
      report(P.status, KVSEL_ERR_BAD_INDEX);
    }
    if (tid < 8) {
      reinterpret_cast<uint4*>(P.idx_k + (size_t(b) * P.max_len + S_old) * kSdDi)[tid] =
          reinterpret_cast<const uint4*>(P.idx_k_new + size_t(b) * kSdDi)[tid];
      __threadfence();  // in L2 before the barrier below: the copies read L2
    }
  }
  for (int i = tid; i < kSdHistBins; i += blockDim.x) s_hist[i] = 0u;
  const int g = lane >> 2, qd = lane & 3;
  // B fragments: indexer head g (zero past Hi), dims permuted as described above
  uint32_t bq[4][2];
  const bool h_ok = g < P.Hi;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint2 v = make_uint2(0u, 0u);
    if (h_ok)
      v = *reinterpret_cast<const uint2*>(P.idx_q + (size_t(b) * P.Hi + g) * kSdDi + 8 * (qd + 4 * (t >> 1)) +
                                          4 * (t & 1));
    bq[t][0] = v.x;
    bq[t][1] = v.y;
  }
  const float w0 = 2 * qd < P.Hi ? P.idx_w[b * P.Hi + 2 * qd] : 0.f;
  const float w1 = 2 * qd + 1 < P.Hi ? P.idx_w[b * P.Hi + 2 * qd + 1] : 0.f;
  float* srow = P.scores + size_t(b) * P.max_len;
  const __nv_bfloat16* kbase = P.idx_k + size_t(b) * P.max_len * kSdDi;
  __syncthreads();  // histogram cleared, the appended key in L2
  // warp w takes the CTA's tiles t0 + w, t0 + w + 8, ...; kSdIdxRing - 1 of them always in flight
  const int nj = t1 - t0 > warp ? (t1 - t0 - warp + kSdIdxWarps - 1) / kSdIdxWarps : 0;
  const uint32_t ring = smem_u32(idx_smem + size_t(kSdHistBins) * 4 + size_t(warp) * kSdIdxRing * kSdIdxTileBytes);
  auto issue = [&](int j) {  // tile j of this warp into its slot (an empty group past the end)
    if (j < nj) {
      const int tile = t0 + warp + j * kSdIdxWarps;
      sd_idx_tile_copy(ring + (j % kSdIdxRing) * kSdIdxTileBytes, kbase + size_t(tile) * 16 * kSdDi,
                       min(16, S - tile * 16), lane);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < kSdIdxRing - 1; ++j) issue(j);
#pragma unroll 1
  for (int j = 0; j < nj; ++j) {
    issue(j + kSdIdxRing - 1);          // into the slot read last iteration
    cp_async_wait<kSdIdxRing - 1>();    // tile j has landed
    __syncwarp();
    // rows g and g + 8, chunks qd and 4 + qd (swizzled: (g + 8) & 7 == g)
    const uint32_t sb = ring + (j % kSdIdxRing) * kSdIdxTileBytes;
    const uint4 ra0 = lds128(sb + g * 128 + ((qd ^ g) << 4));
    const uint4 ra1 = lds128(sb + g * 128 + (((4 + qd) ^ g) << 4));
    const uint4 rb0 = lds128(sb + (g + 8) * 128 + ((qd ^ g) << 4));
    const uint4 rb1 = lds128(sb + (g + 8) * 128 + (((4 + qd) ^ g) << 4));
    __syncwarp();                       // every lane has read the slot before it is refilled
    const int tile = t0 + warp + j * kSdIdxWarps;
    float cc[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16_16816(cc, ra0.x, rb0.x, ra0.y, rb0.y, bq[0][0], bq[0][1]);
    mma_bf16_16816(cc, ra0.z, rb0.z, ra0.w, rb0.w, bq[1][0], bq[1][1]);
    mma_bf16_16816(cc, ra1.x, rb1.x, ra1.y, rb1.y, bq[2][0], bq[2][1]);
    mma_bf16_16816(cc, ra1.z, rb1.z, ra1.w, rb1.w, bq[3][0], bq[3][1]);
    float ia = w0 * fmaxf(cc[0], 0.f) + w1 * fmaxf(cc[1], 0.f);
    float ib = w0 * fmaxf(cc[2], 0.f) + w1 * fmaxf(cc[3], 0.f);
    ia += __shfl_xor_sync(0xffffffffu, ia, 1);
    ia += __shfl_xor_sync(0xffffffffu, ia, 2);
    ib += __shfl_xor_sync(0xffffffffu, ib, 1);
    ib += __shfl_xor_sync(0xffffffffu, ib, 2);
    const int ta = tile * 16 + g, tbk = ta + 8;
    if (qd == 0) {
      if (ta < S) {
        srow[ta] = ia;
        atomicAdd(&s_hist[order_key(ia) >> (32 - kSdHistBits)], 1u);
      }
      if (tbk < S) {
        srow[tbk] = ib;
        atomicAdd(&s_hist[order_key(ib) >> (32 - kSdHistBits)], 1u);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  uint32_t* ghist = P.hist + size_t(b) * kSdHistBins;
  for (int i = tid; i < kSdHistBins; i += blockDim.x) {
    const uint32_t h = s_hist[i];
    if (h) atomicAdd(ghist + i, h);
  }
}

// ---------------------------------------------------------------------------
// Selection.
static_assert(kRkUpMax >= kSdSelSlice && kRkUpMax >= kSdCandCap, "slice keys and candidates fit in ukey");
struct SdSelSmem {
  RowTopkSmem rk;                      // ukey: the slice's keys, then the row's candidate keys; lhist:
                                       // radix select of the last bits; all of it: the whole-row fallback
  int32_t cpos[kSdCandCap];            // the row's candidates in position order: positions
  int32_t crow[kSdCandCap];            // and pool rows for kv head 0
  uint32_t pref[kSdMaxSlices + 1];     // candidate offset of each slice
  uint32_t fin[256];                   // keys of the final sub-bin (their last 8 bits decide)
  int bstar, last, sub, ovf;
  uint32_t above, sub_above, nfin, m, T, need_eq;
};

// The bin holding the kk-th largest of 4096 counts, scanned from the top: thread t holds the
// counts of bins 4095-4t .. 4092-4t in h[0..3].  Writes the bin and the count above it to *bin /
// *above (left alone if the counts hold fewer than kk).  1024 threads.
__device__ __forceinline__ void sd_find_bin(const uint32_t (&h)[4], uint32_t kk, uint32_t* scan_tmp, int* bin,
                                            uint32_t* above_out) {
  const int tid = threadIdx.x;
  const uint32_t v = h[0] + h[1] + h[2] + h[3];
  uint32_t total;
  const uint32_t above = rk_block_excl_scan(v, scan_tmp, total);
  if (above < kk && kk <= above + v) {
    uint32_t run = above;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (run + h[e] >= kk) {
        *bin = kSdHistBins - 1 - 4 * tid - e;
        *above_out = run;
        break;
      }
      run += h[e];
    }
  }
  __syncthreads();
}
__device__ __forceinline__ void sd_load_bins(const uint32_t* hist, uint32_t (&h)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __ldcg(hist + (kSdHistBins - 1 - 4 * int(threadIdx.x) - e));
}

// Per row: every CTA scans a slice of 16K positions, finds from the indexer's
// histogram the bin of the k-th largest score, writes the slice's positions
// in or above that bin (in position order, with their pool rows) to the
// slice's own candidate run, and counts the threshold bin's keys by their
// next 12 bits.  The row's last CTA then knows the sub-bin of the k-th key;
// only the few keys of that sub-bin need their last 8 bits.  It reads the
// candidate runs back in position order, so one block scan gives every kept
// position its place in the ascending output.
__global__ void __launch_bounds__(kSdSelThreads) sd_select_kernel(const SdParams P) {
  extern __shared__ __align__(16) uint8_t sel_smem_raw[];
  SdSelSmem& sm = *reinterpret_cast<SdSelSmem*>(sel_smem_raw);
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");               // scores and histogram are complete
  // The attention may launch once every CTA of this grid has exited or reached the trigger below,
  // which only each row's final CTA does: by then the slice CTAs have left their SMs, so the
  // attention's clusters (eight CTAs in one GPC each) all find room.
  int S;
  if (!sd_len_ok(P, b, S)) return;
  const int k = min(P.top_k, S);
  int32_t* sel = P.sel + size_t(b) * P.top_k;
  int32_t* tko = P.topk_out ? P.topk_out + size_t(b) * P.top_k : nullptr;
  int32_t* srow_out = P.sel_row + size_t(b) * P.top_k;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  uint32_t* ghist = P.hist + size_t(b) * kSdHistBins;
  uint32_t* gsub = P.subhist + size_t(b) * kSdHistBins;
  // a position's pool row for kv head 0 (every kv head adds kvh * page_size), given its page's entry
  const int lg = 4 + P.page_shift;
  auto pool_row = [&](int pos, int phys) {
    if (unsigned(phys) >= unsigned(P.num_pages)) {
      report(P.status, KVSEL_ERR_BAD_INDEX);
      phys = 0;
    }
    return ((phys * P.Hkv) << lg) + (pos & ((1 << lg) - 1));
  };
  auto put = [&](int i, int pos) {
    sel[i] = pos;
    srow_out[i] = pool_row(pos, bt[pos >> lg]);
    if (tko) tko[i] = pos;
  };
  auto finish_row = [&]() {  // the row's histograms and counter back to zero, the count out
    for (int i = tid; i < kSdHistBins; i += kSdSelThreads) {
      ghist[i] = 0u;
      gsub[i] = 0u;
    }
    if (tko)
      for (int i = k + tid; i < P.top_k; i += kSdSelThreads) tko[i] = -1;
    if (tid == 0) {
      P.nsel[b] = k;
      P.row_done[b] = 0u;
    }
  };
  if (k == S) {  // every position is selected: one CTA of the row writes them
    if (c != 0) return;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = tid; i < S; i += kSdSelThreads) put(i, i);
    finish_row();
    return;
  }
  // this CTA's slice: 16 consecutive positions per thread -- one page -- with the histogram bins,
  // the scores and the page's block-table entry all loaded before anything is used; the keys are
  // kept in shared memory (key 0 past the length)
  const int pt = c * kSdSelSlice + 16 * tid;
  uint4* mykeys = reinterpret_cast<uint4*>(sm.rk.ukey + 16 * tid);
  uint32_t h[4];
  sd_load_bins(ghist, h);
  const int phys0 = pt < S ? bt[pt >> lg] : 0;  // the 16 positions lie in one page
  {
    const float* srow = P.scores + size_t(b) * P.max_len;
    if (P.scores_vec && pt + 15 < S) {
      float4 v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __ldcg(reinterpret_cast<const float4*>(srow + pt) + e);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        mykeys[e] = make_uint4(order_key(v[e].x), order_key(v[e].y), order_key(v[e].z), order_key(v[e].w));
    } else {
      uint32_t kk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) kk[e] = pt + e < S ? order_key(__ldcg(srow + pt + e)) : 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) mykeys[e] = make_uint4(kk[4 * e], kk[4 * e + 1], kk[4 * e + 2], kk[4 * e + 3]);
    }
  }
  // the bin holding the k-th largest score (bin 0, every position a candidate, if the counts are short)
  if (tid == 0) {
    sm.bstar = 0;
    sm.above = 0u;
  }
  sd_find_bin(h, uint32_t(k), sm.rk.wtot[0], &sm.bstar, &sm.above);
  const uint32_t lo_key = uint32_t(sm.bstar) << (32 - kSdHistBits);
  const uint32_t bin_hi = (uint32_t(sm.bstar) + 1u) << (32 - kSdHistBits);  // 0 for the top bin
  // candidates (in or above the bin) to this slice's run, in position order; the bin's own keys
  // counted by their next 12 bits
  {
    uint32_t mine = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = mykeys[q];
      const uint32_t kq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool cand = kq[e] >= lo_key && kq[e] != 0u;  // key 0: past the length
        mine += cand ? 1u : 0u;
        if (cand && (bin_hi == 0u || kq[e] < bin_hi)) atomicAdd(gsub + ((kq[e] >> 8) & (kSdHistBins - 1)), 1u);
      }
    }
    uint32_t total;
    uint32_t at = rk_block_excl_scan(mine, sm.rk.wtot[0], total);
    const size_t run = (size_t(b) * P.slices + c) * kSdSliceCap;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = mykeys[q];
      const uint32_t kq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kq[e] >= lo_key && kq[e] != 0u) {
          if (at < uint32_t(kSdSliceCap)) {
            const int pos = pt + 4 * q + e;
            P.cand_key[run + at] = kq[e];
            P.cand_pos[run + at] = pos;
            P.cand_row[run + at] = pool_row(pos, phys0);
          }
          ++at;
        }
    }
    if (tid == 0) P.cand_cnt[size_t(b) * P.slices + c] = total;
  }
  // the last CTA of the row to finish selects
  __syncthreads();
  if (tid == 0) {  // release this CTA's candidates; the last arrival acquires everyone's
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(prev) : "l"(P.row_done + b) : "memory");
    sm.last = prev + 1u == gridDim.x;
  }
  __syncthreads();
  if (!sm.last) return;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // slice offsets and the total (overflow: a slice with more than its capacity), and the sub-bin
  // holding the (k - above)-th best key of the bin; both sets of counts loaded together
  {
    const bool in = tid < P.slices && P.slices <= kSdMaxSlices;
    const uint32_t n = in ? __ldcg(P.cand_cnt + size_t(b) * P.slices + tid) : 0u;
    uint32_t hs[4];
    sd_load_bins(gsub, hs);
    if (tid == 0) {
      sm.ovf = P.slices > kSdMaxSlices;
      sm.sub = 0;
      sm.sub_above = 0u;
      sm.nfin = 0u;
    }
    __syncthreads();
    if (n > uint32_t(kSdSliceCap)) sm.ovf = 1;
    uint32_t total;
    const uint32_t off = rk_block_excl_scan(n, sm.rk.wtot[0], total);
    if (in) sm.pref[tid] = off;
    if (tid == 0) {
      sm.pref[min(P.slices, kSdMaxSlices)] = total;
      sm.m = total;
    }
    sd_find_bin(hs, uint32_t(k) - sm.above, sm.rk.wtot[0], &sm.sub, &sm.sub_above);
  }
  const uint32_t kt = uint32_t(k) - sm.above;  // 1 <= kt <= the bin's count
  const uint32_t m = sm.m;
  if (!sm.ovf && m >= uint32_t(k) && m <= uint32_t(kSdCandCap)) {
    // thread t takes the candidates [t*m/1024, (t+1)*m/1024) in position order: keys to shared
    // memory, the keys of the final sub-bin (they decide by their last 8 bits) to a short list
    constexpr int kPer = kSdCandCap / kSdSelThreads;
    const uint32_t i0 = uint32_t((uint64_t(tid) * m) / kSdSelThreads);
    const uint32_t i1 = uint32_t((uint64_t(tid + 1) * m) / kSdSelThreads);
    const uint32_t p24 = (lo_key >> 8) | uint32_t(sm.sub);
    {
      uint32_t kk[kPer];
      int pp[kPer], rr[kPer];
      int sl = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {  // key, position and pool row, all loads issued together
        const uint32_t i = i0 + j;
        kk[j] = 0u;
        pp[j] = rr[j] = 0;
        if (i < i1) {
          while (sm.pref[sl + 1] <= i) ++sl;  // slices holding no candidate are stepped over
          const size_t src = (size_t(b) * P.slices + sl) * kSdSliceCap + (i - sm.pref[sl]);
          kk[j] = __ldcg(P.cand_key + src);
          pp[j] = __ldcg(P.cand_pos + src);
          rr[j] = __ldcg(P.cand_row + src);
        }
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (i0 + j >= i1) break;
        sm.rk.ukey[i0 + j] = kk[j];
        sm.cpos[i0 + j] = pp[j];
        sm.crow[i0 + j] = rr[j];
        if ((kk[j] >> 8) == p24) {
          const uint32_t at = atomicAdd(&sm.nfin, 1u);
          if (at < 256u) sm.fin[at] = kk[j];
        }
      }
    }
    __syncthreads();
    const uint32_t nf = sm.nfin;
    const uint32_t kf = kt - sm.sub_above;  // 1 <= kf <= nf
    if (nf <= 256u) {  // ranked directly
      if (uint32_t(tid) < nf) {
        const uint32_t f = sm.fin[tid];
        uint32_t gt = 0, eq = 0;
        for (uint32_t x = 0; x < nf; ++x) {
          gt += sm.fin[x] > f;
          eq += sm.fin[x] == f;
        }
        if (gt < kf && kf <= gt + eq) {  // every thread holding this key writes the same values
          sm.T = f;
          sm.need_eq = kf - gt;
        }
      }
    } else {
      uint32_t T, need_eq;
      rk_radix(
          [&](auto&& f) {
            for (int j = 0; j < kPer; ++j) {
              const uint32_t i = i0 + j;
              const uint32_t key = i < i1 ? sm.rk.ukey[i] : 0u;
              const bool live = i < i1 && (key >> 8) == p24;
              f(live ? key : 0u, live);
            }
          },
          7, p24 << 8, kf, sm.rk, T, need_eq);
      if (tid == 0) {
        sm.T = T;
        sm.need_eq = need_eq;
      }
    }
    __syncthreads();
    const uint32_t T = sm.T, need_eq = sm.need_eq;
    // kept: every key above T, and the first need_eq keys equal to it in position order
    uint32_t ng = 0, ne = 0;
    for (uint32_t i = i0; i < i1; ++i) {
      const uint32_t key = sm.rk.ukey[i];
      ng += key > T ? 1u : 0u;
      ne += key == T ? 1u : 0u;
    }
    uint32_t tot;
    const uint32_t ex = rk_block_excl_scan(ng | (ne << 16), sm.rk.wtot[0], tot);
    uint32_t g_before = ex & 0xFFFFu, e_before = ex >> 16;
    for (uint32_t i = i0; i < i1; ++i) {
      const uint32_t key = sm.rk.ukey[i];
      const bool gt = key > T, eq = key == T;
      if (gt || (eq && e_before < need_eq)) {
        const uint32_t o = g_before + min(e_before, need_eq);
        if (o < uint32_t(k)) {
          sel[o] = sm.cpos[i];
          srow_out[o] = sm.crow[i];
          if (tko) tko[o] = sm.cpos[i];
        }
      }
      g_before += gt;
      e_before += eq;
    }
  } else {
    // more candidates than fit (or a very long row): exact top-k over the whole row
    const float* srow = P.scores + size_t(b) * P.max_len;
    const F32RowKeys src{srow, 0, S, (reinterpret_cast<uintptr_t>(srow) & 15u) == 0};
    row_topk<kSdTopkGroups>(src, k, lo_key, sm.rk, put);
  }
  __syncthreads();
  finish_row();
}

// ---------------------------------------------------------------------------
// Thread-block cluster helpers: the splits of one (sequence, kv head) form a
// cluster and merge their partial results through distributed shared memory.
__device__ __forceinline__ void sd_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared variable in cluster CTA `rank`.
__device__ __forceinline__ uint32_t sd_cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float sd_cluster_ld(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t sd_cluster_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}

// ---------------------------------------------------------------------------
// Select for rows of up to kSdCsMaxLen positions, one thread-block cluster of
// kSdCsCtas CTAs per row.  CTA r copies a contiguous chunk of the row's
// scores into its shared memory (warp w: R rounds of 128 consecutive
// positions, 16 bytes a lane) and takes from the indexer's histogram the
// 12-bit bin of the k-th largest key.  One sweep over the chunk then
// compacts, per warp and in position order, the candidates -- keys in or
// above that bin, a few hundred per CTA -- into the warp's own part of the
// buffer; every later step reads the candidates only.  The cluster resolves the k-th key T in two 10-bit radix passes: every CTA adds
// its counts (aggregated per warp) into a histogram in each CTA of the
// cluster through distributed shared memory, and after a cluster barrier each
// CTA finds the same digit in its own copy.  Each CTA counts its kept candidates (above T, and equal to it), pushes
// the totals into every CTA of the cluster, and after a last barrier writes
// its kept positions, in ascending order, straight to the output.  One round
// trip to global memory (the scores, the histogram and the block-table
// entries, issued together) and four cluster barriers, the first while the
// scores are in flight, against the slice
// select's hand-off of candidates through global memory to one final CTA.
constexpr int kSdCsCtas = 8;
constexpr int kSdCsMaxRounds = 8;                                     // 128-position rounds per warp
constexpr int kSdCsChunkMax = 32 * 128 * kSdCsMaxRounds;              // positions per CTA
constexpr int kSdCsMaxLen = kSdCsCtas * kSdCsChunkMax;                // 262144
constexpr int kSdCsDigit = 10;                                        // two passes below the 12-bit bin
constexpr int kSdCsBins = 1 << kSdCsDigit;
static_assert(kSdCsBins == kSdSelThreads, "one radix bin per thread");
static_assert(kSdHistBits + 2 * kSdCsDigit == 32, "the bin and two digits make the whole key");
static_assert(kSdCsChunkMax <= 65536, "chunk positions fit 16 bits");
struct SdCsSmem {
  uint32_t key[kSdCsChunkMax];          // the chunk's scores (raw bits), then each warp's candidate keys
  uint16_t cpos[kSdCsChunkMax];         // the candidates' chunk positions
  int32_t pg[kSdCsChunkMax / 16 + 1];   // block-table entries of the chunk's pages
  uint32_t tot[2][kSdCsBins];           // the two passes' counts over the cluster, added by every CTA
  uint32_t wtot[32];                    // block-scan scratch
  uint32_t wg[32], we[32];              // per-warp kept counts (above / equal to T), then prefixes
  uint32_t allcnt[kSdCsCtas][2];        // every CTA's kept counts, stored here by that CTA
  uint32_t found_d, found_k;
  int bstar;
  uint32_t above;
};

__device__ __forceinline__ void sd_cluster_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sd_cluster_add_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Counts one key per lane into the histogram `hist` of every CTA of the cluster: lanes with the
// same digit add once (a row of equal scores sends thousands of keys to one bin).  Called by the
// whole warp.
__device__ __forceinline__ void sd_warp_count(uint32_t* hist, bool live, uint32_t digit) {
  if (__ballot_sync(0xffffffffu, live)) {
    const uint32_t d = live ? digit : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    if (live && int(threadIdx.x & 31) == __ffs(peers) - 1) {
      const uint32_t n = uint32_t(__popc(peers));
#pragma unroll
      for (int q = 0; q < kSdCsCtas; ++q) sd_cluster_add_u32(sd_cluster_addr(&hist[d], uint32_t(q)), n);
    }
  }
}

__global__ void __launch_bounds__(kSdSelThreads) sd_select_cluster_kernel(const SdParams P) {
  extern __shared__ __align__(16) uint8_t cs_smem_raw[];
  SdCsSmem& sm = *reinterpret_cast<SdCsSmem*>(cs_smem_raw);
  const int r = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // scores and histogram are complete
  // Every early return below is taken by the whole cluster (it depends on the row only), so no
  // CTA is left waiting at a cluster barrier.
  int S;
  if (!sd_len_ok(P, b, S)) return;
  const int k = min(P.top_k, S);
  int32_t* sel = P.sel + size_t(b) * P.top_k;
  int32_t* tko = P.topk_out ? P.topk_out + size_t(b) * P.top_k : nullptr;
  int32_t* srow_out = P.sel_row + size_t(b) * P.top_k;
  const int32_t* bt = P.block_table + size_t(b) * P.max_pages;
  uint32_t* ghist = P.hist + size_t(b) * kSdHistBins;
  const int lg = 4 + P.page_shift;
  auto pool_row = [&](int pos, int phys) {  // the position's pool row for kv head 0
    if (unsigned(phys) >= unsigned(P.num_pages)) {
      report(P.status, KVSEL_ERR_BAD_INDEX);
      phys = 0;
    }
    return ((phys * P.Hkv) << lg) + (pos & ((1 << lg) - 1));
  };
  if (k == S) {  // every position is selected: CTA 0 writes them
    if (r != 0) return;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = tid; i < S; i += kSdSelThreads) {
      sel[i] = i;
      srow_out[i] = pool_row(i, bt[i >> lg]);
      if (tko) tko[i] = i;
    }
    for (int i = tid; i < kSdHistBins; i += kSdSelThreads) ghist[i] = 0u;
    if (tko)
      for (int i = k + tid; i < P.top_k; i += kSdSelThreads) tko[i] = -1;
    if (tid == 0) P.nsel[b] = k;
    return;
  }
  // chunk: R rounds of 128 positions per warp, 32 warps; positions [c0, c0 + lim) are live
  const int R = (S + kSdCsCtas * 32 * 128 - 1) / (kSdCsCtas * 32 * 128);  // <= kSdCsMaxRounds (host)
  const int W = 128 * R, C = 32 * W, c0 = r * C;
  const int lim = max(0, min(C, S - c0));
  const float* srow = P.scores + size_t(b) * P.max_len;
  {
    const uint32_t base = smem_u32(sm.key);
    for (int i = 0; i < R; ++i) {
      const int rel = warp * W + i * 128 + 4 * lane;
      if (P.scores_vec) {  // the row is 16-byte aligned and a multiple of 4 long: 16 bytes a lane
        cp_async16(base + rel * 4, rel < lim ? srow + c0 + rel : srow, rel < lim);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          cp_async4(base + (rel + e) * 4, rel + e < lim ? srow + c0 + rel + e : srow, rel + e < lim);
      }
    }
    cp_async_commit();
  }
  const int pfirst = c0 >> lg;
  const int npg = lim > 0 ? ((c0 + lim - 1) >> lg) - pfirst + 1 : 0;  // <= C / 16 + 1
  for (int i = tid; i < npg; i += kSdSelThreads) sm.pg[i] = bt[pfirst + i];
  uint32_t h[4];
  sd_load_bins(ghist, h);
  // the cluster totals this CTA receives start at zero before any CTA adds to them (the barrier
  // waits while the copies above are in flight)
  sm.tot[0][tid] = 0u;
  sm.tot[1][tid] = 0u;
  if (tid == 0) {
    sm.bstar = 0;
    sm.above = 0u;
  }
  sd_cluster_sync();
  sd_find_bin(h, uint32_t(k), sm.wtot, &sm.bstar, &sm.above);
  const uint32_t bstar = uint32_t(sm.bstar);
  uint32_t kt = uint32_t(k) - sm.above;  // the k-th key's rank among the keys of its bin
  cp_async_wait<0>();
  __syncthreads();  // scores, page entries and cleared histograms visible to the CTA

  // the sweep: each warp's candidates compacted in place, in position order (lane l takes
  // positions 32 e + l of each 128-position round, so a ballot per e gives every candidate its
  // place)
  constexpr int kLoShift = 32 - kSdHistBits;  // 20: bits below the bin
  const uint32_t lo_key = bstar << kLoShift;
  uint32_t* wkey = sm.key + warp * W;
  uint16_t* wpos = sm.cpos + warp * W;
  const unsigned below = (1u << lane) - 1u;
  uint32_t nw = 0;  // the warp's candidates so far
  for (int i = 0; i < R; ++i) {
    const int rel0 = warp * W + i * 128 + lane;
    uint32_t kq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) kq[e] = order_key(__uint_as_float(sm.key[rel0 + 32 * e]));
    __syncwarp();  // the round is read before anyone overwrites it (writes stay below its end)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool cand = rel0 + 32 * e < lim && kq[e] >= lo_key;
      const unsigned m = __ballot_sync(0xffffffffu, cand);
      if (cand) {
        const uint32_t at = nw + __popc(m & below);
        wkey[at] = kq[e];
        wpos[at] = uint16_t(rel0 + 32 * e);
      }
      nw += __popc(m);
    }
  }
  __syncwarp();
  const uint32_t nw_pad = (nw + 31u) & ~31u;

  uint32_t prefix = bstar;
  int shift = kLoShift;  // bits of the key below the prefix
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int dshift = shift - kSdCsDigit;
    uint32_t* hh = sm.tot[pass];
    for (uint32_t j = lane; j < nw_pad; j += 32) {
      const uint32_t key = j < nw ? wkey[j] : 0u;
      sd_warp_count(hh, j < nw && (key >> shift) == prefix, (key >> dshift) & (kSdCsBins - 1));
    }
    sd_cluster_sync();  // every CTA's counts of this pass have arrived
    if (pass == 0 && tid < kSdHistBins / kSdCsCtas)  // every CTA has read the histogram: clear its share
      ghist[r * (kSdHistBins / kSdCsCtas) + tid] = 0u;
    // thread t: digit 1023 - t; the digit holding the kt-th key, from the top
    const int d = kSdCsBins - 1 - tid;
    const uint32_t v = hh[d];
    if (tid == 0) {
      sm.found_d = 0u;
      sm.found_k = 1u;
    }
    uint32_t total;
    const uint32_t above = rk_block_excl_scan(v, sm.wtot, total);
    if (above < kt && kt <= above + v) {
      sm.found_d = uint32_t(d);
      sm.found_k = kt - above;
    }
    __syncthreads();
    prefix = (prefix << kSdCsDigit) | sm.found_d;
    kt = sm.found_k;
    shift = dshift;
  }
  const uint32_t T = prefix, need_eq = kt;  // kept: every key above T and the first need_eq equal to it
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // kept candidates per warp, the warps' prefixes, the CTA's totals to every CTA of the cluster
  {
    uint32_t ng = 0, ne = 0;
    for (uint32_t j = lane; j < nw; j += 32) {
      const uint32_t key = wkey[j];
      ng += key > T ? 1u : 0u;
      ne += key == T ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      ng += __shfl_xor_sync(0xffffffffu, ng, o);
      ne += __shfl_xor_sync(0xffffffffu, ne, o);
    }
    if (lane == 0) {
      sm.wg[warp] = ng;
      sm.we[warp] = ne;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t g0 = sm.wg[lane], e0 = sm.we[lane];
      uint32_t gi = g0, ei = e0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t yg = __shfl_up_sync(0xffffffffu, gi, o), ye = __shfl_up_sync(0xffffffffu, ei, o);
        if (lane >= o) {
          gi += yg;
          ei += ye;
        }
      }
      sm.wg[lane] = gi - g0;
      sm.we[lane] = ei - e0;
      const uint32_t G = __shfl_sync(0xffffffffu, gi, 31), E = __shfl_sync(0xffffffffu, ei, 31);
      if (lane < kSdCsCtas) {  // lane q stores this CTA's totals into CTA q
        sd_cluster_st_u32(sd_cluster_addr(&sm.allcnt[r][0], uint32_t(lane)), G);
        sd_cluster_st_u32(sd_cluster_addr(&sm.allcnt[r][1], uint32_t(lane)), E);
      }
    }
  }
  sd_cluster_sync();  // every CTA's totals are here; no distributed shared memory access follows
  uint32_t before_g = 0, before_e = 0;
  for (int q = 0; q < r; ++q) {
    before_g += sm.allcnt[q][0];
    before_e += sm.allcnt[q][1];
  }
  // emission in position order: a kept key at position p goes to (keys above T before p) +
  // min(keys equal to T before p, need_eq)
  {
    uint32_t g_run = before_g + sm.wg[warp], e_run = before_e + sm.we[warp];
    for (uint32_t j0 = 0; j0 < nw_pad; j0 += 32) {
      const uint32_t j = j0 + lane;
      const uint32_t key = j < nw ? wkey[j] : 0u;
      const bool gt = j < nw && key > T, eq = j < nw && key == T;
      const unsigned mg = __ballot_sync(0xffffffffu, gt), me = __ballot_sync(0xffffffffu, eq);
      const uint32_t gb = g_run + __popc(mg & below), eb = e_run + __popc(me & below);
      if (gt || (eq && eb < need_eq)) {
        const uint32_t o = gb + min(eb, need_eq);
        if (o < uint32_t(k)) {
          const int pos = c0 + int(wpos[j]);
          sel[o] = pos;
          srow_out[o] = pool_row(pos, sm.pg[(pos >> lg) - pfirst]);
          if (tko) tko[o] = pos;
        }
      }
      g_run += __popc(mg);
      e_run += __popc(me);
    }
  }
  if (r == 0 && tid == 0) P.nsel[b] = k;
}

// kWide: 9..16 q heads per kv head (attend_tile_wide)
template <bool kWide>
__global__ void __launch_bounds__(kSdAttnWarps * 32) sd_attn_kernel(const SdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(16) float s_part[kSdPartFloats];  // this split's (M, L, O) of the pair
  __shared__ float s_f[kSdMaxClusterSplits][kSdMaxG];    // each split's max per head, then its merge weight
  __shared__ float s_l[kSdMaxClusterSplits][kSdMaxG];    // each split's sum per head
  float* wo = reinterpret_cast<float*>(smem);  // [4][16][130] merge scratch, over the rings once they are idle
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;  // split = the CTA's rank in its cluster
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G, g = lane >> 2, qd = lane & 3;
  const bool head_ok = g < G, head_ok2 = kWide && g + 8 < G;
  // the q rows and the length are inputs: read while the select finishes (the select writes neither)
  uint32_t qa[8][2], qb[8][2];
  load_q_frags(P.q + (size_t(b) * P.Hq + kvh * G + (head_ok ? g : 0)) * kSdD, head_ok, qd, qa);
  if (kWide) load_q_frags(P.q + (size_t(b) * P.Hq + kvh * G + (head_ok2 ? g + 8 : 0)) * kSdD, head_ok2, qd, qb);
  int S;
  if (!sd_len_ok(P, b, S)) return;  // the whole cluster (one sequence) leaves together
  const int nsel = min(P.top_k, S);
  const int tiles = (nsel + 15) / 16;
  const int t0 = int((long long)split * tiles / P.splits), t1 = int((long long)(split + 1) * tiles / P.splits);
  const int32_t* srow = P.sel_row + size_t(b) * P.top_k;
  const uint32_t wbuf = smem_u32(smem + warp * kSdAttnStages * 8192);
  const int tw0 = t0 + warp;  // this warp's tiles: tw0, tw0 + 4, ... (ordinal j = 0, 1, ...)
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the selection is complete

  TileState st;
  st.init();

  // Pool rows of this warp's tiles j0 .. j0+3, two per lane (lane l: tile j0 + l/16 and
  // j0 + 2 + l/16, key l % 16), all loads issued together; -1 past the selection.
  int ro[2];
  auto load_rows = [&](int j0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tt = tw0 + (j0 + 2 * h + (lane >> 4)) * kSdAttnWarps;
      const int tok = tt * 16 + (lane & 15);
      ro[h] = (tt < t1 && tok < nsel) ? __ldcg(srow + tok) : -1;
    }
  };
  // gather tile ordinal j into stage s: 16 rows of K then 16 of V, 16 x 16-byte units each; the
  // rows' pool positions come from the lanes that loaded them, by shuffles
  auto gather = [&](int j, int s) {
    if ((j & 3) == 0) load_rows(j);
    const int jj = j & 3;
    const int mine = (jj >> 1) ? ro[1] : ro[0];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = lane + 32 * i;
      const int row = c >> 4, u = c & 15;  // row 0..31: K rows 0..15, then V rows
      const int r16 = row & 15;
      const int r = __shfl_sync(0xffffffffu, mine, (jj & 1) * 16 + r16);
      const bool valid = r >= 0;
      const size_t prow = size_t(valid ? r : 0) + (size_t(kvh) << (4 + P.page_shift));
      const __nv_bfloat16* src = (row < 16 ? P.k_pool : P.v_pool) + prow * kSdD + u * 8;
      const uint32_t dst = wbuf + s * 8192 + (row < 16 ? 0 : 4096) + tile_unit_off(r16, u);
      cp_async16(dst, src, valid);
    }
    cp_async_commit();
  };

  // the first kSdAttnStages tiles gathered at once, then one more each time one is consumed (one
  // commit group per tile slot, empty past the end, so the wait below always leaves the newer
  // kSdAttnStages - 1 groups in flight)
#pragma unroll
  for (int j = 0; j < kSdAttnStages; ++j) {
    if (tw0 + j * kSdAttnWarps < t1) gather(j, j);
    else cp_async_commit();
  }
  int s = 0, j = 0;
#pragma unroll 1
  for (int t = tw0; t < t1; t += kSdAttnWarps, ++j) {
    cp_async_wait<kSdAttnStages - 1>();
    __syncwarp();
    const int valid = min(16, nsel - t * 16);
    if (kWide) {
      attend_tile_wide(wbuf + s * 8192, wbuf + s * 8192 + 4096, qa, qb, valid, P.scale_log2, st, head_ok, head_ok2);
    } else {
      float x0, x1, x2, x3;
      attend_tile(wbuf + s * 8192, wbuf + s * 8192 + 4096, qa, valid, P.scale_log2, st, x0, x1, x2, x3);
    }
    __syncwarp();
    if (t + kSdAttnStages * kSdAttnWarps < t1) gather(j + kSdAttnStages, s);
    else cp_async_commit();
    s = s + 1 == kSdAttnStages ? 0 : s + 1;
  }
  cp_async_wait<0>();
  // the next step's indexer may launch now: it waits for this grid before touching anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();  // every warp is done with its ring: the merge scratch may overwrite it
  merge_warps_to_slot<kSdAttnWarps, kWide>(st, wo, s_part, G);
  sd_cluster_sync();  // every split's partial is in its shared memory
  // merge weights: every split's (max, sum) per head fetched at once, then combined per head
  const int ns = P.splits;
  if (tid < ns * G) {
    const int sp = tid / G, gg = tid % G;
    s_f[sp][gg] = sd_cluster_ld(sd_cluster_addr(&s_part[gg], sp));
    s_l[sp][gg] = sd_cluster_ld(sd_cluster_addr(&s_part[kSdMaxG + gg], sp));
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, s_f[sp][tid]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int sp = 0; sp < ns; ++sp)
        if (s_f[sp][tid] != -INFINITY) L += s_l[sp][tid] * exp2f(s_f[sp][tid] - M);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int sp = 0; sp < ns; ++sp) {
      const float ms = s_f[sp][tid];
      s_f[sp][tid] = (M != -INFINITY && ms != -INFINITY) ? exp2f(ms - M) * inv : 0.f;
    }
  }
  __syncthreads();
  // this split's share of the pair's G x 128 outputs
  const int E = G * kSdD;
  const int e1 = (split + 1) * E / ns;
  for (int idx = split * E / ns + tid; idx < e1; idx += kSdAttnWarps * 32) {
    const int gg = idx / kSdD, dd = idx % kSdD;
    float pv[kSdMaxClusterSplits];  // every split's value issued before any is used
#pragma unroll
    for (int sp = 0; sp < kSdMaxClusterSplits; ++sp)
      pv[sp] = sp < ns ? sd_cluster_ld(sd_cluster_addr(&s_part[2 * kSdMaxG + gg * kSdD + dd], uint32_t(sp))) : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int sp = 0; sp < kSdMaxClusterSplits; ++sp)
      if (sp < ns) acc += s_f[sp][gg] * pv[sp];
    const size_t oi = (size_t(b) * P.Hq + size_t(kvh) * G + gg) * kSdD + dd;
    if (P.out_f32) static_cast<float*>(P.out)[oi] = acc;
    else static_cast<__nv_bfloat16*>(P.out)[oi] = __float2bfloat16_rn(acc);
  }
  sd_cluster_sync();  // no CTA leaves while another still reads its partial
  // the last (sequence, kv head) cluster of a sequence publishes its length: every CTA of the
  // sequence has read the old one by then
  if (split == 0 && tid == 0) {
    __threadfence();
    if (atomicAdd(P.seq_cnt + b, 1u) + 1u == unsigned(P.Hkv)) {
      P.seq_cnt[b] = 0u;
      P.seq_lens[b] = S;
    }
  }
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct SdWs {
  size_t scores, hist, cnt, ckey, cpos, crow, sel, srow, nsel, total;
};
SdWs sd_ws_layout(int batch, int max_len, int top_k, bool own_scores) {
  SdWs w;
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.scores = own_scores ? take(size_t(batch) * max_len * 4) : 0;
  const size_t slices = size_t((max_len + kSdSelSlice - 1) / kSdSelSlice);
  w.hist = take(size_t(batch) * kSdHistBins * 4 * 2);        // the indexer's histogram, then the sub-bins
  w.cnt = take(size_t(batch) * (slices + 2) * 4);            // per-slice candidates, CTAs done, kv heads merged
  w.ckey = take(size_t(batch) * slices * kSdSliceCap * 4);
  w.cpos = take(size_t(batch) * slices * kSdSliceCap * 4);
  w.crow = take(size_t(batch) * slices * kSdSliceCap * 4);
  w.sel = take(size_t(batch) * top_k * 4);
  w.srow = take(size_t(batch) * top_k * 4);
  w.nsel = take(size_t(batch) * 4);
  w.total = off;
  return w;
}
}  // namespace

extern "C" size_t kvsel_sparse_decode_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                                int top_k, int with_scores_out) {
  if (!kv || batch < 1 || max_len < 1 || top_k < 1 || kv->num_kv_heads < 1) return 0;
  return sd_ws_layout(batch, max_len, top_k, with_scores_out == 0).total;
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
  if (kv->head_dim != kSdD || page_shift_of(kv->page_size) < 0)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16, 32, 64, 128 or 256 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (G > kSdMaxG) return fail(KVSEL_ERR_UNSUPPORTED, fn + "at most 16 q heads per kv head");
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
  const SdWs L = sd_ws_layout(batch, max_len, top_k, scores_out == nullptr);
  if (max_len > kSdMaxLen) return fail(KVSEL_ERR_UNSUPPORTED, fn + "max_len must be <= 2^28");
  if ((long long)kv->num_pages * Hkv * kv->page_size >= (1LL << 31))
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "num_pages * num_kv_heads * page_size must be below 2^31");
  if (!aligned(kv->k_pool, 16) || !aligned(kv->v_pool, 16) || !aligned(q, 16) || !aligned(idx_k, 16) ||
      !aligned(idx_q, 8) || (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(idx_k_new, 16))))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pools, q, k_new, v_new, idx_k, idx_k_new must be 16-byte aligned");
  if (!workspace || !aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "a 256-byte aligned workspace is required");
  if (ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace too small: need " + std::to_string(L.total));

  const int sms = sm_count();
  // indexer: two CTAs per SM over the whole batch, each a contiguous run of one row's tiles
  const int idx_ctas = std::max(1, (2 * sms + batch - 1) / batch);
  // attention: one wave at two CTAs per SM
  const int tiles_max = (std::min(top_k, max_len) + 15) / 16;
  int splits = std::max(1, (2 * sms) / (batch * Hkv));
  splits = std::min(splits, std::max(1, (tiles_max + 3) / 4));
  splits = std::min(splits, kSdMaxClusterSplits);

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
  P.page_shift = page_shift_of(kv->page_size);
  const int slices = (max_len + kSdSelSlice - 1) / kSdSelSlice;
  P.hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  P.subhist = P.hist + size_t(batch) * kSdHistBins;
  P.cand_cnt = reinterpret_cast<unsigned*>(ws + L.cnt);
  P.row_done = P.cand_cnt + size_t(batch) * slices;
  P.seq_cnt = P.row_done + batch;
  P.slices = slices;
  P.cand_key = reinterpret_cast<uint32_t*>(ws + L.ckey);
  P.cand_pos = reinterpret_cast<int32_t*>(ws + L.cpos);
  P.cand_row = reinterpret_cast<int32_t*>(ws + L.crow);
  P.sel = reinterpret_cast<int32_t*>(ws + L.sel);
  P.sel_row = reinterpret_cast<int32_t*>(ws + L.srow);
  P.nsel = reinterpret_cast<int32_t*>(ws + L.nsel);
  P.topk_out = topk_out;
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
  P.idx_ctas = idx_ctas;
  P.scores_vec = (max_len % 4 == 0) && aligned(P.scores, 16);
  P.splits = splits;
  P.appended = k_new ? 1 : 0;
  P.out_f32 = out_dtype == KVSEL_F32;
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    cudaError_t e0 = smem_limit_once(reinterpret_cast<const void*>(sd_attn_kernel<false>), int(kSdAttnSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(sd_attn_kernel<true>), int(kSdAttnSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(sd_index_kernel), int(kSdIdxSmem));
    if (e0 == cudaSuccess)
      e0 = smem_limit_once(reinterpret_cast<const void*>(sd_select_kernel), int(sizeof(SdSelSmem)));
    if (e0 == cudaSuccess)
      e0 = smem_limit_once(reinterpret_cast<const void*>(sd_select_cluster_kernel), int(sizeof(SdCsSmem)));
    if (e0 != cudaSuccess) return cuda_fail(e0, "kvsel_sparse_decode (attribute)");
  }
  cudaError_t e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // set per launch below
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.stream = st;
  // Every kernel may launch while its predecessor runs (programmatic launch) and waits for it
  // before reading its results; each predecessor lets the next one in as early as that is useful.
#define KVSEL_SD_LAUNCH(name, kernel, grid, block, smem, nattr)          \
  cfg.gridDim = grid;                                                    \
  cfg.blockDim = dim3(block);                                            \
  cfg.dynamicSmemBytes = smem;                                           \
  cfg.attrs = nattr ? attr : nullptr;                                    \
  cfg.numAttrs = nattr;                                                  \
  trace_before(name, st);                                                \
  e = cudaLaunchKernelEx(&cfg, kernel, P);                               \
  trace_after(st);                                                       \
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_sparse_decode (" name ")");
  KVSEL_SD_LAUNCH("sd_index", sd_index_kernel, dim3(idx_ctas, batch), kSdIdxWarps * 32, kSdIdxSmem, 1)
  if (max_len <= kSdCsMaxLen) {  // a row's select: one cluster of kSdCsCtas CTAs
    attr[1].val.clusterDim.x = unsigned(kSdCsCtas);
    KVSEL_SD_LAUNCH("sd_select", sd_select_cluster_kernel, dim3(kSdCsCtas, batch), kSdSelThreads,
                    sizeof(SdCsSmem), 2)
  } else {  // longer rows: slices of 16K positions hand their candidates to the row's last CTA
    KVSEL_SD_LAUNCH("sd_select", sd_select_kernel, dim3(slices, batch), kSdSelThreads, sizeof(SdSelSmem), 1)
  }
  attr[1].val.clusterDim.x = unsigned(splits);  // the attention's splits of a pair: one cluster
  if (G > 8) {
    KVSEL_SD_LAUNCH("sd_attn", sd_attn_kernel<true>, dim3(splits, Hkv, batch), kSdAttnWarps * 32, kSdAttnSmem, 2)
  } else {
    KVSEL_SD_LAUNCH("sd_attn", sd_attn_kernel<false>, dim3(splits, Hkv, batch), kSdAttnWarps * 32, kSdAttnSmem, 2)
  }
#undef KVSEL_SD_LAUNCH
  return KVSEL_OK;
}
