// SnapKV prefill selection (sm_103a).
//
// What it computes ("From sliding window to attention-guided eviction" §4.3,
// steps 2-5): for every layer and kv head, the last W prompt queries of the
// group's G q heads (the observation window, G*W rows) attend causally to the
// prompt: window query i sits at position S - W + i and sees keys 0..S-W+i.
// The vote of a prefix key j < S - W is the sum over all G*W rows of its
// softmax weight; the vote is max-pooled (stride 1, window clipped to the
// prefix) and the top keep_k prefix positions (ties to the lower position)
// plus the window itself are kept, in ascending order.
//
// Kernels (four launches per call, all layers at once):
//   snap_qk_kernel<1>  row softmax statistics: every CTA streams a chunk of a
//                      (layer, kv head)'s K pages (TMA, 8-stage ring) and 8
//                      warps each run 32 window rows against every page with
//                      mma.sync (S = Q K^T), keeping an online (max, sum) per
//                      row; partial statistics per chunk.
//   snap_qk_kernel<2>  votes: the same contraction again (K comes back from
//                      L2 or HBM), weights exp2(s - M_row) / L_row from the
//                      merged statistics, summed over the warp's rows with
//                      shuffles and over the 8 warps in shared memory.
//   snap_pool_kernel   max-pool of the votes into order keys (tiles of 1024
//                      positions staged in shared memory with their halo).
//   snap_select_kernel exact top-keep_k of the pooled keys per (layer, kv
//                      head) with row_topk, window appended.
#include "common.cuh"
#include "row_topk.cuh"
#include "umma.cuh"

namespace kvsel {

constexpr int kSnD = 128;
constexpr int kSnPage = 16;
constexpr int kSnMaxRows = 256;          // G * W <= 256
constexpr int kSnMaxChunks = 64;
constexpr int kSnSelGroups = 8;           // register-resident rows: prefix <= 32768
constexpr int kSnPoolTile = 1024;
constexpr int kSnMaxHalf = 16;            // pool kernel <= 33

struct SnapParams {
  const int32_t* block_table;  // [L][max_pages]
  const __nv_bfloat16* q_obs;  // [L][Hq][W][128]
  float* stats;                // [L*Hkv][chunks][rows][2]
  float* vote;                 // [L*Hkv][S - W]
  int32_t* keep_out;           // [L*Hkv][keep_k + W]
  uint32_t* pool_key;          // [L*Hkv][pool_stride]: order keys of the pooled votes
  int pool_stride;
  int* status;
  int L, Hq, Hkv, G, W, rows, S, max_pages, num_pages, chunks, keep_k, pool_half;
  float scale_log2;
};

// ---------------------------------------------------------------------------
// The contraction on the 5th-generation tensor cores.  One CTA per (chunk of
// keys, layer x kv head); warp 0 streams the chunk's K pages by TMA into a
// ring of 128-key tiles, warp 1 issues tcgen05.mma (one elected thread) into
// a double-buffered TMEM accumulator, warps 2..5 read the accumulator back
// (tcgen05.ld) and do the softmax work.
//   pass 1 (row statistics): D[rows x keys] = Q K^T, rows on the M side in
//           one or two 128-row tiles; each epilogue thread owns one row and
//           keeps its online (max, sum) in the log2 domain;
//   pass 2 (votes): D[keys x rows] = K Q^T, keys on the M side; each
//           epilogue thread owns one key and sums its weights over the rows
//           directly, so the vote needs no cross-thread reduction.
// ---------------------------------------------------------------------------
constexpr int kTcKeys = 128;                          // keys per MMA tile (8 pages)
constexpr int kTcStages = 4;                          // K tiles in flight
constexpr int kTcTileBytes = 2 * kTcKeys * 128;       // two 64-column slabs
constexpr int kTcQRows = 256;
constexpr int kTcQBytes = 2 * kTcQRows * 128;
constexpr int kTcEpiPerQ = 4;                         // epilogue warps per TMEM lane quarter
constexpr int kTcEpiWarps = 4 * kTcEpiPerQ;
constexpr int kTcThreads = (2 + kTcEpiWarps) * 32;    // producer, MMA issuer, epilogue
constexpr uint32_t kTcCols = 512;                     // TMEM columns: 2 accumulators x 256
struct TcLayout {
  static constexpr size_t q = 0;
  static constexpr size_t ring = q + kTcQBytes;
  static constexpr size_t bars = ring + size_t(kTcStages) * kTcTileBytes;  // full, empty, acc_full, acc_empty
  static constexpr size_t tmem = bars + (2 * kTcStages + 4) * 8;
  static constexpr size_t stat = tmem + 16;        // [kTcQRows] f32: pass 2 row offsets C = M - log2(1/L)
  static constexpr size_t xch = stat + size_t(kTcQRows) * 4;  // partial exchange between a quarter's warps
  static constexpr size_t total = xch + size_t(2) * 2 * kTcEpiPerQ * 4 * 32 * 4;
};
constexpr size_t kTcSmem = TcLayout::total + 1024;
static_assert(kSnMaxRows <= kTcQRows, "window rows fit in the Q tile");

// 2^x on the special-function unit (ex2.approx, relative error ~2^-22; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int kPass>
__global__ void __launch_bounds__(kTcThreads, 1)
snap_tc_kernel(const __grid_constant__ CUtensorMap tmK, const SnapParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + TcLayout::q;
  uint8_t* sK = smem + TcLayout::ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TcLayout::bars);
  uint64_t* empty = full + kTcStages;
  uint64_t* acc_full = empty + kTcStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_word = reinterpret_cast<uint32_t*>(smem + TcLayout::tmem);
  float* sStat = reinterpret_cast<float*>(smem + TcLayout::stat);

  const int chunk = blockIdx.x, pair = blockIdx.y;
  const int layer = pair / P.Hkv, kvh = pair % P.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = P.rows;
  const int Pfx = P.S - P.W;
  const int span = kPass == 1 ? P.S : Pfx;  // keys this pass needs
  const int npages = (span + kSnPage - 1) / kSnPage;
  const int pb = int((long long)chunk * npages / P.chunks);
  const int pe = int((long long)(chunk + 1) * npages / P.chunks);
  const int key0 = pb * kSnPage, key1 = min(span, pe * kSnPage);
  const int ntiles = (pe - pb + 7) / 8;

  // ---- Q rows of this (layer, kv head), 128-byte swizzled K-major; zero padding ----
  {
    const __nv_bfloat16* qbase = P.q_obs + ((size_t(layer) * P.Hq + kvh * P.G) * P.W) * kSnD;
    for (int idx = tid; idx < kTcQRows * 16; idx += kTcThreads) {
      const int r = idx >> 4, ch = idx & 15, slab = ch >> 3, c = ch & 7;
      const uint4 v = r < R ? reinterpret_cast<const uint4*>(qbase + size_t(r) * kSnD)[ch] : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sQ + slab * (kTcQRows * 128) + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
  }
  if (kPass == 2) {
    // merged row statistics: M = max over chunks, 1/L with L = sum l * 2^(m - M)
    const float* st = P.stats + size_t(pair) * P.chunks * R * 2;
    for (int r = tid; r < R; r += kTcThreads) {
      float M = -INFINITY;
      for (int c = 0; c < P.chunks; ++c) M = fmaxf(M, st[(size_t(c) * R + r) * 2]);
      float Lr = 0.f;
      if (M != -INFINITY)
        for (int c = 0; c < P.chunks; ++c) {
          const float m = st[(size_t(c) * R + r) * 2];
          if (m != -INFINITY) Lr += st[(size_t(c) * R + r) * 2 + 1] * exp2f(m - M);
        }
      // weight = 2^(s - M) / L = 2^(s - C) with C = M + log2(L); rows without keys weigh 0
      sStat[r] = (M != -INFINITY && Lr > 0.f) ? M + __log2f(Lr) : INFINITY;
    }
    for (int r = R + tid; r < kTcQRows; r += kTcThreads) sStat[r] = INFINITY;  // padding rows weigh 0
  }
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), kTcEpiWarps * 32);
    }
    mbar_fence_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q stores -> tensor-core reads
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_word), kTcCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_word;

  if (warp == 0) {
    // ---- producer: up to 8 pages per tile, two 64-column boxes per page.  The
    // lanes resolve block-table entries 32 pages (4 tiles) at a time, one group
    // ahead, so no dependent table load sits between two tiles' TMA issues ----
    const uint64_t pol = l2_policy_evict_first();
    const int32_t* bt = P.block_table + size_t(layer) * P.max_pages;
    const int n = pe - pb;
    auto resolve = [&](int i) -> int {  // TMA row of chunk-local page i (0 past the end)
      if (i >= n) return 0;
      int phys = bt[pb + i];
      if (unsigned(phys) >= unsigned(P.num_pages)) {
        report(P.status, KVSEL_ERR_BAD_INDEX);
        phys = 0;
      }
      return (phys * P.Hkv + kvh) * kSnPage;
    };
    int y_cur = resolve(lane), y_next = resolve(32 + lane);
    bool stop = false;
#pragma unroll 1
    for (int t = 0; t < ntiles && !stop; ++t) {
      const int pl = 8 * t;  // chunk-local first page of the tile
      if (t > 0 && (pl & 31) == 0) {
        y_cur = y_next;
        y_next = resolve(pl + 32 + lane);
      }
      int ys[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ys[i] = __shfl_sync(0xffffffffu, y_cur, (pl & 31) + i);
      const int s = t % kTcStages;
      bool ok = true;
      if (lane == 0 && t >= kTcStages) ok = mbar_wait(smem_u32(&empty[s]), ((t / kTcStages) + 1) & 1, P.status);
      stop = !__shfl_sync(0xffffffffu, ok, 0);
      if (!stop && lane == 0) {
        const int np = min(8, n - pl);
        const uint32_t dst = smem_u32(sK + s * kTcTileBytes);
        const uint32_t bar = smem_u32(&full[s]);
        mbar_expect_tx(bar, uint32_t(np) * 4096u);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < np) {
            tma_load_2d(dst + i * 2048, &tmK, 0, ys[i], bar, pol);
            tma_load_2d(dst + kTcKeys * 128 + i * 2048, &tmK, 64, ys[i], bar, pol);
          }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      const int nMt = (R + 127) / 128;
      const int Npad = (R + 31) & ~31;  // zero-padded rows up to whole 32-column loads
      const uint32_t idesc = kPass == 1 ? umma_idesc_bf16_f32(128, kTcKeys) : umma_idesc_bf16_f32(128, Npad);
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kTcStages, buf = t & 1;
        if (!mbar_wait(smem_u32(&full[s]), (t / kTcStages) & 1, P.status)) break;
        if (t >= 2 && !mbar_wait(smem_u32(&acc_empty[buf]), ((t >> 1) + 1) & 1, P.status)) break;
        tc_fence_after();
        const uint32_t kt = smem_u32(sK + s * kTcTileBytes);
        const uint32_t qt = smem_u32(sQ);
        if (kPass == 1) {
          for (int mt = 0; mt < nMt; ++mt)
            for (int k = 0; k < 8; ++k) {
              const uint32_t koff = uint32_t(k >> 2) * (kTcKeys * 128) + uint32_t(k & 3) * 32;
              const uint32_t qoff = uint32_t(k >> 2) * (kTcQRows * 128) + uint32_t(mt) * (128 * 128) + uint32_t(k & 3) * 32;
              umma_bf16(tbase + uint32_t(buf) * 256 + uint32_t(mt) * 128, umma_desc_sw128(qt + qoff),
                        umma_desc_sw128(kt + koff), idesc, k > 0);
            }
        } else {
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = uint32_t(k >> 2) * (kTcKeys * 128) + uint32_t(k & 3) * 32;
            const uint32_t qoff = uint32_t(k >> 2) * (kTcQRows * 128) + uint32_t(k & 3) * 32;
            umma_bf16(tbase + uint32_t(buf) * 256, umma_desc_sw128(kt + koff), umma_desc_sw128(qt + qoff), idesc,
                      k > 0);
          }
        }
        umma_commit(smem_u32(&empty[s]));     // the K tile may be overwritten once these MMAs are done
        umma_commit(smem_u32(&acc_full[buf]));
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: kTcEpiPerQ warps share TMEM lane quarter w & 3, each a
    // part of the columns (pass 1: keys of a tile, pass 2: window rows) ----
    const int quarter = warp & 3, part = (warp - 2) >> 2;
    const int tl = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const int nMt = (R + 127) / 128;
    float* xch = reinterpret_cast<float*>(smem + TcLayout::xch);
    auto qsync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + quarter), "n"(32 * kTcEpiPerQ) : "memory"); };
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int limit[2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) limit[mt] = Pfx + ((mt * 128 + tl) % P.W);
    float* vrow = P.vote + size_t(pair) * Pfx;
    const float sc = P.scale_log2;
    bool dead = false;  // a wait ran out: keep the trip count (named barriers), skip the waits
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t) {
      const int buf = t & 1;
      if (!dead) dead = !mbar_wait(smem_u32(&acc_full[buf]), (t >> 1) & 1, P.status);
      tc_fence_after();
      const int kt0 = (pb + 8 * t) * kSnPage;
      const uint32_t acc = tbase + lane_addr + uint32_t(buf) * 256;
      if (kPass == 1) {
        // a tile wholly inside [key0, key1) and the prefix needs no mask
        const bool plain = kt0 >= key0 && kt0 + kTcKeys <= key1 && kt0 + kTcKeys <= Pfx;
        constexpr int kCols = kTcKeys / kTcEpiPerQ;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          if (mt >= nMt) break;
#pragma unroll 1
          for (int c0 = part * kCols; c0 < (part + 1) * kCols; c0 += 32) {
            float v[32];
            tmem_ld32(acc + uint32_t(mt) * 128 + uint32_t(c0), v);
            if (!plain) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int key = kt0 + c0 + i;
                if (!(key >= key0 && key < key1 && key <= limit[mt])) v[i] = -INFINITY;
              }
            }
            float mx = -INFINITY;  // raw logits (the scale is positive)
#pragma unroll
            for (int i = 0; i < 32; i += 2) mx = max3(mx, v[i], v[i + 1]);
            const float m_new = fmaxf(m_run[mt], mx * sc);
            if (m_new != -INFINITY) {
              float sum = 0.f;
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                sum += fast_exp2(fmaf(v[i], sc, -m_new)) + fast_exp2(fmaf(v[i + 1], sc, -m_new)) +
                       fast_exp2(fmaf(v[i + 2], sc, -m_new)) + fast_exp2(fmaf(v[i + 3], sc, -m_new));
              }
              l_run[mt] = l_run[mt] * fast_exp2(m_run[mt] - m_new) + sum;
              m_run[mt] = m_new;
            }
          }
        }
      } else {
        const int nchunks = ((R + 31) & ~31) / 32;
        const int cbeg = nchunks * part / kTcEpiPerQ, cend = nchunks * (part + 1) / kTcEpiPerQ;
        float vote = 0.f;
#pragma unroll 1
        for (int ci = cbeg; ci < cend; ++ci) {
          const int c0 = ci * 32;
          float v[32];
          tmem_ld32(acc + uint32_t(c0), v);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 C = *reinterpret_cast<const float4*>(sStat + c0 + i);  // +inf past the rows
            vote += fast_exp2(fmaf(v[i], sc, -C.x)) + fast_exp2(fmaf(v[i + 1], sc, -C.y)) +
                    fast_exp2(fmaf(v[i + 2], sc, -C.z)) + fast_exp2(fmaf(v[i + 3], sc, -C.w));
          }
        }
        float* xb = xch + ((buf * kTcEpiPerQ + part) * 4 + quarter) * 32;  // [parity][part][quarter][32]
        xb[lane] = vote;
        qsync();
        if (part == 0) {
          const int key = kt0 + tl;
          float sum = 0.f;
#pragma unroll
          for (int q = 0; q < kTcEpiPerQ; ++q) sum += xch[((buf * kTcEpiPerQ + q) * 4 + quarter) * 32 + lane];
          if (key >= key0 && key < key1) vrow[key] = sum;
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&acc_empty[buf]));
    }
    if (kPass == 1) {
      // merge the parts' (m, l) per row, then write this chunk's statistics
      float* xm = xch;                                   // [2 mt][part][quarter][32]
      float* xl = xch + 2 * kTcEpiPerQ * 4 * 32;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        xm[((mt * kTcEpiPerQ + part) * 4 + quarter) * 32 + lane] = m_run[mt];
        xl[((mt * kTcEpiPerQ + part) * 4 + quarter) * 32 + lane] = l_run[mt];
      }
      qsync();
      if (part == 0) {
        float* st = P.stats + (size_t(pair) * P.chunks + chunk) * R * 2;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          float M = -INFINITY;
#pragma unroll
          for (int q = 0; q < kTcEpiPerQ; ++q) M = fmaxf(M, xm[((mt * kTcEpiPerQ + q) * 4 + quarter) * 32 + lane]);
          float Lr = 0.f;
          if (M != -INFINITY)
#pragma unroll
            for (int q = 0; q < kTcEpiPerQ; ++q) {
              const float m = xm[((mt * kTcEpiPerQ + q) * 4 + quarter) * 32 + lane];
              if (m != -INFINITY) Lr += xl[((mt * kTcEpiPerQ + q) * 4 + quarter) * 32 + lane] * fast_exp2(m - M);
            }
          if (mt < nMt && mt * 128 + tl < R) {
            st[(mt * 128 + tl) * 2] = M;
            st[(mt * 128 + tl) * 2 + 1] = Lr;
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTcCols);
  }
}

// Stride-1 max-pool of the votes over [j - pool_half, j + pool_half] clipped
// to the prefix, stored as order keys; one tile of 1024 positions per CTA.
__global__ void __launch_bounds__(kSnPoolTile) snap_pool_kernel(const SnapParams P) {
  __shared__ float tile[kSnPoolTile + 2 * kSnMaxHalf];
  const int pair = blockIdx.y, tid = threadIdx.x;
  const int Pfx = P.S - P.W, h = P.pool_half;
  const int j0 = blockIdx.x * kSnPoolTile;
  const float* vrow = P.vote + size_t(pair) * Pfx;
  for (int i = tid; i < kSnPoolTile + 2 * h; i += kSnPoolTile) {
    const int j = j0 - h + i;
    tile[i] = (j >= 0 && j < Pfx) ? __ldcg(vrow + j) : -INFINITY;
  }
  __syncthreads();
  const int j = j0 + tid;
  if (j < Pfx) {
    float mx = tile[tid];
    for (int t = 1; t <= 2 * h; ++t) mx = fmaxf(mx, tile[tid + t]);
    P.pool_key[size_t(pair) * P.pool_stride + j] = order_key(mx);
  }
}

// Exact top-keep_k of the pooled votes, then the window, ascending.
__global__ void __launch_bounds__(kRkThreads) snap_select_kernel(const SnapParams P) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  RowTopkSmem& sm = *reinterpret_cast<RowTopkSmem*>(tk_smem);
  const int pair = blockIdx.x, tid = threadIdx.x;
  const int Pfx = P.S - P.W;
  const int nk = P.keep_k + P.W;
  int32_t* keep = P.keep_out + size_t(pair) * nk;
  if (Pfx <= P.keep_k) {  // nothing to evict: every position, then -1 padding
    for (int i = tid; i < nk; i += kRkThreads) keep[i] = i < P.S ? i : -1;
    return;
  }
  const uint32_t* krow = P.pool_key + size_t(pair) * P.pool_stride;
  const U32RowKeys src{krow, 0, Pfx, (reinterpret_cast<uintptr_t>(krow) & 15u) == 0};
  row_topk<kSnSelGroups>(src, P.keep_k, 0u, sm, [&](int i, int rel) { keep[i] = rel; });
  for (int i = tid; i < P.W; i += kRkThreads) keep[P.keep_k + i] = Pfx + i;
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct SnWs {
  size_t stats, vote, pool, total;
  int pool_stride;
};
SnWs sn_ws_layout(int L, int Hkv, int rows, int S, int W, int chunks, bool own_vote) {
  SnWs w;
  size_t off = kStatusBytes;
  w.stats = off;
  off = align_up(off + size_t(L) * Hkv * chunks * rows * 2 * 4, 256);
  w.vote = off;
  if (own_vote) off = align_up(off + size_t(L) * Hkv * std::max(S - W, 1) * 4, 256);
  w.pool = off;
  w.pool_stride = int(align_up(size_t(std::max(S - W, 1)), 4));
  off = align_up(off + size_t(L) * Hkv * w.pool_stride * 4, 256);
  w.total = off;
  return w;
}
// Key chunks per (layer, kv head): one CTA per SM, so pick the count that
// minimises waves x 128-key tiles per CTA (fewer chunks on ties).
int sn_chunks(int L, int Hkv, int S) {
  const int tiles = ((S + kSnPage - 1) / kSnPage + 7) / 8;
  const long long pairs = (long long)L * Hkv, sms = sm_count();
  int best = 1;
  long long best_cost = -1;
  for (int c = 1; c <= std::min(kSnMaxChunks, tiles); ++c) {
    const long long cost = ((pairs * c + sms - 1) / sms) * ((tiles + c - 1) / c);
    if (best_cost < 0 || cost < best_cost) {
      best = c;
      best_cost = cost;
    }
  }
  return best;
}
}  // namespace

extern "C" size_t kvsel_snapkv_select_workspace(const kvsel_paged_kv* kv, int num_layers, int seq_len,
                                                int obs_window, int with_vote_out) {
  if (!kv || num_layers < 1 || seq_len < 1 || obs_window < 1 || kv->num_kv_heads < 1 ||
      kv->num_q_heads % kv->num_kv_heads != 0)
    return 0;
  const int rows = kv->num_q_heads / kv->num_kv_heads * obs_window;
  return sn_ws_layout(num_layers, kv->num_kv_heads, rows, seq_len, obs_window, kSnMaxChunks,
                      with_vote_out == 0).total;
}

extern "C" kvsel_status kvsel_snapkv_select(const kvsel_paged_kv* kv, const int32_t* block_table,
                                            int max_pages, int num_layers, int seq_len, const void* q_obs,
                                            int obs_window, float scale, int pool_kernel, int keep_k,
                                            int32_t* keep_out, float* vote_out, void* workspace,
                                            size_t ws_bytes, void* stream) {
  const std::string fn = "kvsel_snapkv_select: ";
  if (!kv || !kv->k_pool) return fail(KVSEL_ERR_INVALID_ARG, fn + "the K pool is required");
  if (kv->head_dim != kSnD || kv->page_size != kSnPage)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "only head_dim 128 and page_size 16 are implemented");
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_q_heads must be a positive multiple of num_kv_heads");
  const int Hkv = kv->num_kv_heads, Hq = kv->num_q_heads, G = Hq / Hkv;
  if (!block_table || !q_obs || !keep_out || num_layers < 1 || max_pages < 1 || obs_window < 1 ||
      seq_len < obs_window || keep_k < 1)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "block_table, q_obs, keep_out required; 1 <= obs_window <= "
                                            "seq_len, keep_k >= 1");
  const int rows = G * obs_window;
  if (rows > kSnMaxRows)
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "(q heads per kv head) * obs_window must be <= 256");
  if (seq_len >= (1 << 28))
    return fail(KVSEL_ERR_UNSUPPORTED, fn + "seq_len must be < 2^28");
  if (!(scale > 0.f))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "scale must be positive");
  if (pool_kernel < 1 || pool_kernel % 2 == 0 || pool_kernel / 2 > kSnMaxHalf)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "pool_kernel must be odd, 1..33");
  if ((seq_len + kSnPage - 1) / kSnPage > max_pages)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "seq_len exceeds max_pages * 16");
  if (kv->num_pages < 1 || (long long)kv->num_pages * Hkv * kSnPage >= (1LL << 31))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "num_pages * num_kv_heads * 16 must be in [1, 2^31)");
  if (!aligned(kv->k_pool, 16) || !aligned(q_obs, 16))
    return fail(KVSEL_ERR_INVALID_ARG, fn + "K pool and q_obs must be 16-byte aligned");
  const int chunks = sn_chunks(num_layers, Hkv, seq_len);
  const SnWs L = sn_ws_layout(num_layers, Hkv, rows, seq_len, obs_window, kSnMaxChunks, vote_out == nullptr);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "workspace missing, misaligned or smaller than " +
                                           std::to_string(L.total));
  CUtensorMap tmK;
  if (!encode_bf16_2d(&tmK, kv->k_pool, kSnD, uint64_t(kv->num_pages) * Hkv * kSnPage, kSnD * 2, 64, kSnPage))
    return fail(KVSEL_ERR_CUDA, fn + "tensor-map encode failed");

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SnapParams P;
  P.block_table = block_table;
  P.q_obs = static_cast<const __nv_bfloat16*>(q_obs);
  P.stats = reinterpret_cast<float*>(ws + L.stats);
  P.vote = vote_out ? vote_out : reinterpret_cast<float*>(ws + L.vote);
  P.keep_out = keep_out;
  P.pool_key = reinterpret_cast<uint32_t*>(ws + L.pool);
  P.pool_stride = L.pool_stride;
  P.status = reinterpret_cast<int*>(ws);
  P.L = num_layers;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.W = obs_window;
  P.rows = rows;
  P.S = seq_len;
  P.max_pages = max_pages;
  P.num_pages = kv->num_pages;
  P.chunks = chunks;
  P.keep_k = keep_k;
  P.pool_half = pool_kernel / 2;
  P.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    cudaError_t e0 = smem_limit_once(reinterpret_cast<const void*>(snap_tc_kernel<1>), int(kTcSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(snap_tc_kernel<2>), int(kTcSmem));
    if (e0 == cudaSuccess)
      e0 = smem_limit_once(reinterpret_cast<const void*>(snap_select_kernel), int(sizeof(RowTopkSmem)));
    if (e0 != cudaSuccess) return cuda_fail(e0, "kvsel_snapkv_select (attribute)");
  }
  const dim3 grid(chunks, num_layers * Hkv);
  cudaError_t e;
  trace_before("snap_stats", st);
  snap_tc_kernel<1><<<grid, kTcThreads, kTcSmem, st>>>(tmK, P);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (stats launch)");
  if (seq_len > obs_window) {
    trace_before("snap_vote", st);
    snap_tc_kernel<2><<<grid, kTcThreads, kTcSmem, st>>>(tmK, P);
    e = cudaGetLastError();
    trace_after(st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (vote launch)");
  }
  if (seq_len - obs_window > keep_k) {
    trace_before("snap_pool", st);
    snap_pool_kernel<<<dim3((seq_len - obs_window + kSnPoolTile - 1) / kSnPoolTile, num_layers * Hkv),
                       kSnPoolTile, 0, st>>>(P);
    e = cudaGetLastError();
    trace_after(st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (pool launch)");
  }
  trace_before("snap_select", st);
  snap_select_kernel<<<num_layers * Hkv, kRkThreads, sizeof(RowTopkSmem), st>>>(P);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (select launch)");
  return KVSEL_OK;
}
