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
// Two variants of the same section: the GQA union (each q head picks its own
// top-k from its own pooled vote; the kv head keeps the union of its heads'
// picks, then the window) and the cold-start seed (for every kept key, the
// attention the G*W window rows gave it, window keys included causally: the
// accumulator H2O would hold had the last W prompt tokens been decoded one
// at a time with the same queries).
//
// Kernels (three launches per call, all layers at once; four for the union):
//   snap_tc_kernel<1>  row softmax statistics: every CTA streams a chunk of a
//                      (layer, kv head)'s K pages by TMA into a 4-tile ring,
//                      one thread issues tcgen05.mma (S = Q K^T into TMEM),
//                      16 epilogue warps keep an online (max, sum) per row;
//                      partial statistics per chunk.
//   snap_tc_kernel<2>  votes: the same contraction again with keys on the M
//                      side (K comes back from L2 or HBM), weights
//                      exp2(s - M_row) / L_row from the merged statistics,
//                      each epilogue thread summing one key's row weights.
//   snap_tc_kernel<3>  the union variant's per-q-head votes instead of <2>.
//   snap_select_kernel exact top-keep_k of the max-pooled votes per (layer,
//                      kv head) with row_topk, the pool taken as the row is
//                      loaded; window appended, seeds gathered; per q head
//                      for the union variant.
//   snap_union_kernel  union variant: bitmap of the group's picks, emitted in
//                      ascending order with the window and the seeds.
#include "common.cuh"
#include "row_topk.cuh"
#include "umma.cuh"

namespace kvsel {

constexpr int kSnD = 128;
constexpr int kSnPage = 16;
constexpr int kSnMaxRows = 256;          // G * W <= 256
constexpr int kSnMaxChunks = 64;
constexpr int kSnSelGroups = 8;           // register-resident rows: prefix <= 32768
constexpr int kSnMaxHalf = 16;            // max-pool window (pool_kernel) <= 33

struct SnapParams {
  const int32_t* block_table;  // [L][max_pages]
  const __nv_bfloat16* q_obs;  // [L][Hq][W][128]
  float* stats;                // [L*Hkv][chunks][rows][2]
  float* vote;                 // [L*Hkv][S - W]; the union variant: [L*Hq][S - W]
  float* wvote;                // window keys' attention (the seed of keys S-W..S-1), rows as vote x [W]
  int32_t* keep_out;           // [L*Hkv][keep_cap]
  int32_t* keep_count;         // [L*Hkv] or null
  int32_t* head_keep;          // union variant: [L*Hq][keep_k] per-head picks
  uint32_t* bitmap;            // union variant: [L*Hkv][nwords] marks of the group's picks
  float* seed;                 // kept keys' seeds (null: none), at layer * seed_ls + kv head * seed_hs
  long long seed_ls, seed_hs;
  int* status;
  int L, Hq, Hkv, G, W, rows, S, max_pages, num_pages, chunks, keep_k, pool_half;
  int union_mode, keep_cap, vote_span, nwords;  // vote_span: S with seeds (window keys too), else S - W
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
//           directly, so the vote needs no cross-thread reduction;
//   pass 3 (per-head votes, union variant): the same product; the four
//           epilogue warps of a lane quarter split the group's heads and sum
//           each head's W columns apart.
// With seeds the vote passes also cover the window keys, whose weights are
// masked causally per (key, row).
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
  const int span = kPass == 1 ? P.S : P.vote_span;  // keys this pass needs
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
  if (kPass >= 2) {
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
      } else if (kPass == 2) {
        const int nchunks = ((R + 31) & ~31) / 32;
        const int cbeg = nchunks * part / kTcEpiPerQ, cend = nchunks * (part + 1) / kTcEpiPerQ;
        // a tile reaching the window keys masks row r of window key Pfx + kw unless r % W >= kw
        const bool wtile = kt0 + kTcKeys > Pfx;
        const int kw = kt0 + tl - Pfx;
        float vote = 0.f;
#pragma unroll 1
        for (int ci = cbeg; ci < cend; ++ci) {
          const int c0 = ci * 32;
          float v[32];
          tmem_ld32(acc + uint32_t(c0), v);
          if (!wtile) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 C = *reinterpret_cast<const float4*>(sStat + c0 + i);  // +inf past the rows
              vote += fast_exp2(fmaf(v[i], sc, -C.x)) + fast_exp2(fmaf(v[i + 1], sc, -C.y)) +
                      fast_exp2(fmaf(v[i + 2], sc, -C.z)) + fast_exp2(fmaf(v[i + 3], sc, -C.w));
            }
          } else {
            int rw = c0 % P.W;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float C = rw >= kw ? sStat[c0 + i] : INFINITY;
              vote += fast_exp2(fmaf(v[i], sc, -C));
              rw = rw + 1 == P.W ? 0 : rw + 1;
            }
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
          if (key >= key0 && key < key1) {
            if (key < Pfx) vrow[key] = sum;
            else P.wvote[size_t(pair) * P.W + (key - Pfx)] = sum;
          }
        }
      } else {
        // per-q-head votes: this warp's heads g0..g1-1, W columns each, no exchange
        const int g0 = P.G * part / kTcEpiPerQ, g1 = P.G * (part + 1) / kTcEpiPerQ;
        const int key = kt0 + tl, kw = key - Pfx;
        const bool wtile = kt0 + kTcKeys > Pfx;
#pragma unroll 1
        for (int g = g0; g < g1; ++g) {
          const int lo = g * P.W, hi = lo + P.W;
          const bool whole = !wtile && (lo & 31) == 0 && (P.W & 31) == 0;  // 32-column loads inside the head
          float vote = 0.f;
#pragma unroll 1
          for (int c0 = lo & ~31; c0 < hi; c0 += 32) {
            float v[32];
            tmem_ld32(acc + uint32_t(c0), v);
            if (whole) {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 C = *reinterpret_cast<const float4*>(sStat + c0 + i);
                vote += fast_exp2(fmaf(v[i], sc, -C.x)) + fast_exp2(fmaf(v[i + 1], sc, -C.y)) +
                        fast_exp2(fmaf(v[i + 2], sc, -C.z)) + fast_exp2(fmaf(v[i + 3], sc, -C.w));
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int r = c0 + i;
                const bool in = r >= lo && r < hi && r - lo >= kw;  // kw < 0 for prefix keys
                vote += fast_exp2(fmaf(v[i], sc, in ? -sStat[r] : -INFINITY));
              }
            }
          }
          if (key >= key0 && key < key1) {
            const size_t vr = size_t(layer) * P.Hq + size_t(kvh) * P.G + g;
            if (key < Pfx) P.vote[vr * Pfx + key] = vote;
            else P.wvote[vr * P.W + (key - Pfx)] = vote;
          }
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

// Keys of the max-pooled votes of one row, pooled as they are loaded: key(j)
// = order key of max(p[j - h .. j + h]) with the window clipped to the prefix
// [0, n) (stride 1).  row_topk loads a row once when it fits its registers
// (prefix <= 32768), so the pooled row is never stored.  load4 must be called
// by all 32 lanes of a warp together (row_topk's sweep does): for h <= 4 a
// lane loads its own four votes and takes the halo from the neighbouring
// lanes' (lane i - 1 / i + 1 when they hold positions rel - 4 / rel + 4, else
// it loads them itself).
struct PooledVoteKeys {
  const float* p;
  int lo, n, h;
  __device__ __forceinline__ float at(int j) const { return (j >= 0 && j < n) ? __ldcg(p + j) : -INFINITY; }
  __device__ __forceinline__ uint32_t key(int j, float m) const { return (j >= lo && j < n) ? order_key(m) : 0u; }
  __device__ __forceinline__ uint32_t load1(int rel) const {
    if (rel < lo || rel >= n) return 0u;
    float m = -INFINITY;
#pragma unroll 8
    for (int t = -h; t <= h; ++t) m = fmaxf(m, at(rel + t));
    return order_key(m);
  }
  __device__ __forceinline__ uint4 load4(int rel) const {
    float w[12];  // positions rel - 4 .. rel + 7
#pragma unroll
    for (int i = 0; i < 4; ++i) w[4 + i] = at(rel + i);
    if (h <= 4) {
      const int rl = __shfl_up_sync(0xffffffffu, rel, 1), rr = __shfl_down_sync(0xffffffffu, rel, 1);
      const int lane = threadIdx.x & 31;
      const bool left = lane > 0 && rl == rel - 4, right = lane < 31 && rr == rel + 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = __shfl_up_sync(0xffffffffu, w[4 + i], 1), b = __shfl_down_sync(0xffffffffu, w[4 + i], 1);
        w[i] = left ? a : at(rel - 4 + i);
        w[8 + i] = right ? b : at(rel + 4 + i);
      }
      float m[4];
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        m[o] = w[4 + o];
#pragma unroll
        for (int i = 0; i < 12; ++i) {
          const int d = i - 4 - o;  // offset of position rel - 4 + i from output rel + o
          if (d != 0 && d >= -4 && d <= 4 && (d < 0 ? -d : d) <= h) m[o] = fmaxf(m[o], w[i]);
        }
      }
      return make_uint4(key(rel, m[0]), key(rel + 1, m[1]), key(rel + 2, m[2]), key(rel + 3, m[3]));
    }
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
    for (int t = -h; t <= h + 3; ++t) {  // wide pools: position rel + t feeds outputs o with |t - o| <= h
      const float x = at(rel + t);
      if (t <= h) m0 = fmaxf(m0, x);
      if (t >= 1 - h && t <= h + 1) m1 = fmaxf(m1, x);
      if (t >= 2 - h && t <= h + 2) m2 = fmaxf(m2, x);
      if (t >= 3 - h) m3 = fmaxf(m3, x);
    }
    return make_uint4(key(rel, m0), key(rel + 1, m1), key(rel + 2, m2), key(rel + 3, m3));
  }
};

// Seed of key j of vote row vr (j < S: the prefix from the votes, the window
// from the window-key sums).
__device__ __forceinline__ float snap_seed_of(const SnapParams& P, size_t vr, int Pfx, int j) {
  return j < Pfx ? P.vote[vr * Pfx + j] : P.wvote[vr * P.W + (j - Pfx)];
}

// Exact top-keep_k of the pooled votes, then the window, ascending; the
// union variant stores each q head's picks for snap_union_kernel instead.
__global__ void __launch_bounds__(kRkThreads) snap_select_kernel(const SnapParams P) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  RowTopkSmem& sm = *reinterpret_cast<RowTopkSmem*>(tk_smem);
  const int row = blockIdx.x, tid = threadIdx.x;
  const int Pfx = P.S - P.W;
  const PooledVoteKeys src{P.vote + size_t(row) * Pfx, 0, Pfx, P.pool_half};
  if (P.union_mode) {  // launched only when Pfx > keep_k
    int32_t* hk = P.head_keep + size_t(row) * P.keep_k;
    row_topk<kSnSelGroups>(src, P.keep_k, 0u, sm, [&](int i, int rel) { hk[i] = rel; });
    return;
  }
  const int nk = P.keep_cap;
  int32_t* keep = P.keep_out + size_t(row) * nk;
  float* sd = P.seed ? P.seed + (row / P.Hkv) * P.seed_ls + (row % P.Hkv) * P.seed_hs : nullptr;
  if (Pfx <= P.keep_k) {  // nothing to evict: every position, then -1 padding
    for (int i = tid; i < nk; i += kRkThreads) {
      keep[i] = i < P.S ? i : -1;
      if (sd) sd[i] = i < P.S ? snap_seed_of(P, size_t(row), Pfx, i) : 0.f;
    }
    if (tid == 0 && P.keep_count) P.keep_count[row] = P.S;
    return;
  }
  row_topk<kSnSelGroups>(src, P.keep_k, 0u, sm, [&](int i, int rel) { keep[i] = rel; });
  if (sd) {
    __syncthreads();  // the picks are this block's own global stores
    for (int i = tid; i < P.keep_k; i += kRkThreads) sd[i] = P.vote[size_t(row) * Pfx + keep[i]];
  }
  for (int i = tid; i < P.W; i += kRkThreads) {
    keep[P.keep_k + i] = Pfx + i;
    if (sd) sd[P.keep_k + i] = P.wvote[size_t(row) * P.W + i];
  }
  if (tid == 0 && P.keep_count) P.keep_count[row] = P.keep_k + P.W;
}

// Union variant, one CTA per (layer, kv head): mark the G heads' picks in a
// bitmap, then emit the marked positions in ascending order (a block scan of
// the words' popcounts per round of kUnThreads words), the window after them,
// -1 padding up to keep_cap; seeds summed over the group's vote rows.
constexpr int kUnThreads = 512;
__global__ void __launch_bounds__(kUnThreads) snap_union_kernel(const SnapParams P) {
  __shared__ int wsum[kUnThreads / 32];
  __shared__ int s_base;
  const int pair = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int layer = pair / P.Hkv, kvh = pair % P.Hkv;
  const int Pfx = P.S - P.W, nk = P.keep_cap;
  const size_t vr0 = size_t(layer) * P.Hq + size_t(kvh) * P.G;  // the group's first vote row
  int32_t* keep = P.keep_out + size_t(pair) * nk;
  float* sd = P.seed ? P.seed + layer * P.seed_ls + kvh * P.seed_hs : nullptr;
  auto seed = [&](int j) {
    float a = 0.f;
#pragma unroll 4
    for (int g = 0; g < P.G; ++g) a += snap_seed_of(P, vr0 + g, Pfx, j);
    return a;
  };
  int count;
  if (Pfx <= P.keep_k) {  // every head keeps its whole prefix
    count = Pfx;
    for (int i = tid; i < Pfx; i += kUnThreads) {
      keep[i] = i;
      if (sd) sd[i] = seed(i);
    }
  } else {
    uint32_t* bits = P.bitmap + size_t(pair) * P.nwords;
    const int nw = (Pfx + 31) >> 5;
    for (int w = tid; w < nw; w += kUnThreads) bits[w] = 0u;
    __syncthreads();
    const int32_t* hk = P.head_keep + vr0 * P.keep_k;
    for (int i = tid; i < P.G * P.keep_k; i += kUnThreads) {
      const int x = hk[i];
      if (unsigned(x) < unsigned(Pfx)) atomicOr(bits + (x >> 5), 1u << (x & 31));
      else report(P.status, KVSEL_ERR_BAD_INDEX);
    }
    __syncthreads();
    if (tid == 0) s_base = 0;
    for (int w0 = 0; w0 < nw; w0 += kUnThreads) {
      const int w = w0 + tid;
      uint32_t word = w < nw ? __ldcg(bits + w) : 0u;
      const int c = __popc(word);
      int incl = c;  // warp inclusive scan
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        int t = lane < kUnThreads / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, t, o);
          if (lane >= o) t += y;
        }
        if (lane < kUnThreads / 32) wsum[lane] = t;  // inclusive totals per warp
      }
      __syncthreads();
      int off = s_base + (warp > 0 ? wsum[warp - 1] : 0) + incl - c;
      while (word) {
        const int b = __ffs(word) - 1;
        word &= word - 1;
        keep[off++] = w * 32 + b;
      }
      __syncthreads();
      if (tid == 0) s_base += wsum[kUnThreads / 32 - 1];
      __syncthreads();
    }
    count = s_base;
    if (sd) {  // seeds in a pass of their own, four entries per thread at a time (this block's own stores)
      for (int o0 = tid; o0 < count; o0 += 4 * kUnThreads) {
        int j[4];
        float a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) j[u] = o0 + u * kUnThreads < count ? keep[o0 + u * kUnThreads] : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = 0.f;
        for (int g = 0; g < P.G; ++g) {
          const float* vg = P.vote + (vr0 + g) * Pfx;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (j[u] >= 0) a[u] += __ldcg(vg + j[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j[u] >= 0) sd[o0 + u * kUnThreads] = a[u];
      }
    }
  }
  for (int i = tid; i < nk - count; i += kUnThreads) {
    const int o = count + i;
    keep[o] = i < P.W ? Pfx + i : -1;
    if (sd) sd[o] = i < P.W ? seed(Pfx + i) : 0.f;
  }
  if (tid == 0 && P.keep_count) P.keep_count[pair] = count + P.W;
}

}  // namespace kvsel

using namespace kvsel;
using namespace kvsel_host;

namespace {
struct SnWs {
  size_t stats, vote, wvote, hkeep, bitmap, total;
  int nwords;
};
// vote rows: one per (layer, kv head), or per (layer, q head) for the union
SnWs sn_ws_layout(int L, int Hkv, int Hq, int rows, int S, int W, int chunks, bool own_vote, bool union_mode) {
  SnWs w;
  const size_t vrows = size_t(L) * (union_mode ? Hq : Hkv);
  const size_t pfx = size_t(std::max(S - W, 1));
  size_t off = kStatusBytes;
  w.stats = off;
  off = align_up(off + size_t(L) * Hkv * chunks * rows * 2 * 4, 256);
  w.vote = off;
  if (own_vote) off = align_up(off + vrows * pfx * 4, 256);
  w.wvote = off;
  off = align_up(off + vrows * W * 4, 256);
  w.hkeep = off;
  if (union_mode) off = align_up(off + vrows * pfx * 4, 256);  // keep_k < S - W whenever it is used
  w.bitmap = off;
  w.nwords = int((pfx + 31) / 32);
  if (union_mode) off = align_up(off + size_t(L) * Hkv * w.nwords * 4, 256);
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

extern "C" size_t kvsel_snapkv_select_ex_workspace(const kvsel_paged_kv* kv, int num_layers, int seq_len,
                                                   int obs_window, int with_vote_out, int mode) {
  if (!kv || num_layers < 1 || seq_len < 1 || obs_window < 1 || kv->num_kv_heads < 1 ||
      kv->num_q_heads % kv->num_kv_heads != 0 || (mode != KVSEL_SNAP_GROUP_SUM && mode != KVSEL_SNAP_HEAD_UNION))
    return 0;
  const int rows = kv->num_q_heads / kv->num_kv_heads * obs_window;
  return sn_ws_layout(num_layers, kv->num_kv_heads, kv->num_q_heads, rows, seq_len, obs_window, kSnMaxChunks,
                      with_vote_out == 0, mode == KVSEL_SNAP_HEAD_UNION).total;
}

extern "C" size_t kvsel_snapkv_select_workspace(const kvsel_paged_kv* kv, int num_layers, int seq_len,
                                                int obs_window, int with_vote_out) {
  return kvsel_snapkv_select_ex_workspace(kv, num_layers, seq_len, obs_window, with_vote_out,
                                          KVSEL_SNAP_GROUP_SUM);
}

extern "C" kvsel_status kvsel_snapkv_select(const kvsel_paged_kv* kv, const int32_t* block_table,
                                            int max_pages, int num_layers, int seq_len, const void* q_obs,
                                            int obs_window, float scale, int pool_kernel, int keep_k,
                                            int32_t* keep_out, float* vote_out, void* workspace,
                                            size_t ws_bytes, void* stream) {
  return kvsel_snapkv_select_ex(kv, block_table, max_pages, num_layers, seq_len, q_obs, obs_window, scale,
                                pool_kernel, keep_k, nullptr, keep_out, vote_out, workspace, ws_bytes, stream);
}

extern "C" kvsel_status kvsel_snapkv_select_ex(const kvsel_paged_kv* kv, const int32_t* block_table,
                                               int max_pages, int num_layers, int seq_len, const void* q_obs,
                                               int obs_window, float scale, int pool_kernel, int keep_k,
                                               const kvsel_snap_options* opt, int32_t* keep_out,
                                               float* vote_out, void* workspace, size_t ws_bytes,
                                               void* stream) {
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
  const int mode = opt ? opt->mode : KVSEL_SNAP_GROUP_SUM;
  if (mode != KVSEL_SNAP_GROUP_SUM && mode != KVSEL_SNAP_HEAD_UNION)
    return fail(KVSEL_ERR_INVALID_ARG, fn + "mode must be KVSEL_SNAP_GROUP_SUM or KVSEL_SNAP_HEAD_UNION");
  const bool uni = mode == KVSEL_SNAP_HEAD_UNION;
  const long long cap = (uni ? (long long)G * keep_k : (long long)keep_k) + obs_window;
  if (cap >= (1LL << 31)) return fail(KVSEL_ERR_INVALID_ARG, fn + "keep capacity must be < 2^31");
  float* seed = opt ? opt->seed_out : nullptr;
  if (seed) {
    const long long ls = opt->seed_layer_stride, hs = opt->seed_head_stride;
    if (hs < cap || (num_layers > 1 && ls < hs * Hkv))
      return fail(KVSEL_ERR_INVALID_ARG, fn + "seed strides must give every (layer, kv head) its own row of "
                                              "the keep capacity");
  }
  const int chunks = sn_chunks(num_layers, Hkv, seq_len);
  const SnWs L = sn_ws_layout(num_layers, Hkv, Hq, rows, seq_len, obs_window, kSnMaxChunks, vote_out == nullptr,
                              uni);
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
  P.wvote = reinterpret_cast<float*>(ws + L.wvote);
  P.keep_count = opt ? opt->keep_count : nullptr;
  P.head_keep = reinterpret_cast<int32_t*>(ws + L.hkeep);
  P.bitmap = reinterpret_cast<uint32_t*>(ws + L.bitmap);
  P.seed = seed;
  P.seed_ls = seed ? opt->seed_layer_stride : 0;
  P.seed_hs = seed ? opt->seed_head_stride : 0;
  P.union_mode = uni ? 1 : 0;
  P.keep_cap = int(cap);
  P.vote_span = seed ? seq_len : seq_len - obs_window;
  P.nwords = L.nwords;
  const int Pfx = seq_len - obs_window;
  const int vrows = num_layers * (uni ? Hq : Hkv);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    cudaError_t e0 = smem_limit_once(reinterpret_cast<const void*>(snap_tc_kernel<1>), int(kTcSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(snap_tc_kernel<2>), int(kTcSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(snap_tc_kernel<3>), int(kTcSmem));
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
  if (Pfx > 0 || seed) {  // votes (and the window keys' sums when seeding)
    trace_before("snap_vote", st);
    if (uni) snap_tc_kernel<3><<<grid, kTcThreads, kTcSmem, st>>>(tmK, P);
    else snap_tc_kernel<2><<<grid, kTcThreads, kTcSmem, st>>>(tmK, P);
    e = cudaGetLastError();
    trace_after(st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (vote launch)");
  }
  if (!uni || Pfx > keep_k) {
    trace_before("snap_select", st);
    snap_select_kernel<<<vrows, kRkThreads, sizeof(RowTopkSmem), st>>>(P);
    e = cudaGetLastError();
    trace_after(st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (select launch)");
  }
  if (uni) {
    trace_before("snap_union", st);
    snap_union_kernel<<<num_layers * Hkv, kUnThreads, 0, st>>>(P);
    e = cudaGetLastError();
    trace_after(st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (union launch)");
  }
  return KVSEL_OK;
}
