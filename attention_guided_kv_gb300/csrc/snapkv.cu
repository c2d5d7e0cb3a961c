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

namespace kvsel {

constexpr int kSnD = 128;
constexpr int kSnPage = 16;
constexpr int kSnStages = 8;
constexpr int kSnStageBytes = 4096;       // one K page: two 2 KB swizzled halves
constexpr int kSnWarps = 8;               // consumer warps: 32 window rows each
constexpr int kSnThreads = (kSnWarps + 1) * 32;
constexpr int kSnMaxRows = kSnWarps * 32; // G * W <= 256
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

__device__ __forceinline__ uint32_t sn_tile_off(int key, int u) {
  return (u >> 3) * 2048 + key * 128 + ((((u & 7) ^ (key & 7))) << 4);
}

template <int kPass>
__global__ void __launch_bounds__(kSnThreads, 1)
snap_qk_kernel(const __grid_constant__ CUtensorMap tmK, const SnapParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSnStages * kSnStageBytes);
  uint64_t* empty = full + kSnStages;
  float* vacc = reinterpret_cast<float*>(empty + kSnStages);  // [stages][16]
  int* vcnt = reinterpret_cast<int*>(vacc + kSnStages * 16);  // [stages]
  float* sStat = reinterpret_cast<float*>(vcnt + kSnStages);  // [rows][2] merged (pass 2)

  const int chunk = blockIdx.x, pair = blockIdx.y;
  const int layer = pair / P.Hkv, kvh = pair % P.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Pfx = P.S - P.W;                      // prefix length
  const int span = kPass == 1 ? P.S : Pfx;        // keys this pass needs
  const int npages = (span + kSnPage - 1) / kSnPage;
  const int pb = int((long long)chunk * npages / P.chunks);
  const int pe = int((long long)(chunk + 1) * npages / P.chunks);
  const int n = pe - pb;

  if (tid == 0) {
    for (int s = 0; s < kSnStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kSnWarps);
    }
    mbar_fence_init();
  }
  for (int i = tid; i < kSnStages * 16; i += kSnThreads) vacc[i] = 0.f;
  if (tid < kSnStages) vcnt[tid] = 0;
  if (kPass == 2) {
    // merged row statistics: M = max over chunks, 1/L with L = sum l * 2^(m - M)
    const float* st = P.stats + size_t(pair) * P.chunks * P.rows * 2;
    for (int r = tid; r < P.rows; r += kSnThreads) {
      float M = -INFINITY;
      for (int c = 0; c < P.chunks; ++c) M = fmaxf(M, st[(size_t(c) * P.rows + r) * 2]);
      float Lr = 0.f;
      if (M != -INFINITY)
        for (int c = 0; c < P.chunks; ++c) {
          const float m = st[(size_t(c) * P.rows + r) * 2];
          if (m != -INFINITY) Lr += st[(size_t(c) * P.rows + r) * 2 + 1] * exp2f(m - M);
        }
      sStat[r * 2] = M;
      sStat[r * 2 + 1] = Lr > 0.f ? 1.f / Lr : 0.f;
    }
  }
  __syncthreads();

  if (warp == kSnWarps) {
    // producer: one K page of this (layer, kv head) per stage
    if (lane == 0 && n > 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int32_t* bt = P.block_table + size_t(layer) * P.max_pages;
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int s = i % kSnStages;
        if (i >= kSnStages && !mbar_wait(smem_u32(&empty[s]), ((i / kSnStages) + 1) & 1, P.status)) break;
        int phys = bt[pb + i];
        if (unsigned(phys) >= unsigned(P.num_pages)) {
          report(P.status, KVSEL_ERR_BAD_INDEX);
          phys = 0;
        }
        const int y = (phys * P.Hkv + kvh) * kSnPage;
        const uint32_t dst = smem_u32(smem + s * kSnStageBytes);
        const uint32_t bar = smem_u32(&full[s]);
        mbar_expect_tx(bar, kSnStageBytes);
        tma_load_2d(dst, &tmK, 0, y, bar, pol);
        tma_load_2d(dst + 2048, &tmK, 64, y, bar, pol);
      }
    }
    return;
  }

  // ---- consumers: warp w owns rows [32w, 32w + 32) as two m16 tiles ----
  const int g = lane >> 2, qd = lane & 3, mi = lane >> 3, r8 = lane & 7;
  const bool active = warp * 32 < P.rows;
  int rowid[4];                  // rows of this lane: [mt][g or g+8]
  bool rowok[4];
  int limit[4];                  // last visible key of the row (causal)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    rowid[k] = warp * 32 + (k >> 1) * 16 + g + (k & 1) * 8;
    rowok[k] = rowid[k] < P.rows;
    limit[k] = Pfx + (rowid[k] % P.W);
  }
  uint32_t qa[2][8][4];
  {
    const __nv_bfloat16* qbase = P.q_obs + ((size_t(layer) * P.Hq + kvh * P.G) * P.W) * kSnD;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint32_t* r0 = reinterpret_cast<const uint32_t*>(qbase + size_t(rowok[2 * mt] ? rowid[2 * mt] : 0) * kSnD);
      const uint32_t* r1 = reinterpret_cast<const uint32_t*>(qbase + size_t(rowok[2 * mt + 1] ? rowid[2 * mt + 1] : 0) * kSnD);
#pragma unroll
      for (int kt = 0; kt < 8; ++kt) {
        qa[mt][kt][0] = rowok[2 * mt] ? r0[(16 * kt + 2 * qd) >> 1] : 0u;
        qa[mt][kt][1] = rowok[2 * mt + 1] ? r1[(16 * kt + 2 * qd) >> 1] : 0u;
        qa[mt][kt][2] = rowok[2 * mt] ? r0[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
        qa[mt][kt][3] = rowok[2 * mt + 1] ? r1[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
      }
    }
  }
  float m_run[4], l_run[4], Mr[4], Ir[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    m_run[k] = -INFINITY;
    l_run[k] = 0.f;
    Mr[k] = kPass == 2 && rowok[k] ? sStat[rowid[k] * 2] : 0.f;
    Ir[k] = kPass == 2 && rowok[k] ? sStat[rowid[k] * 2 + 1] : 0.f;
  }
  float* vrow = P.vote + size_t(pair) * Pfx;

#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    const int s = i % kSnStages;
    if (!mbar_wait(smem_u32(&full[s]), (i / kSnStages) & 1, P.status)) break;
    const int key0 = (pb + i) * kSnPage;
    if (active) {
      const uint32_t kb = smem_u32(smem + s * kSnStageBytes);
      float acc[2][2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
#pragma unroll
      for (int kt = 0; kt < 8; ++kt) {
        const int key = (mi >> 1) * 8 + r8;
        const int uu = 2 * kt + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + sn_tile_off(key, uu), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_bf16_16816(acc[mt][0], qa[mt][kt][0], qa[mt][kt][1], qa[mt][kt][2], qa[mt][kt][3], b0, b1);
          mma_bf16_16816(acc[mt][1], qa[mt][kt][0], qa[mt][kt][1], qa[mt][kt][2], qa[mt][kt][3], b2, b3);
        }
      }
      // acc[mt][nt][e]: row (mt, e >> 1), key key0 + 8 nt + 2 qd + (e & 1)
      if (kPass == 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int mt = k >> 1, hr = k & 1;
          float x[4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = key0 + 8 * nt + 2 * qd + e;
              const bool vis = rowok[k] && key < P.S && key <= limit[k];
              x[nt * 2 + e] = vis ? acc[mt][nt][hr * 2 + e] * P.scale_log2 : -INFINITY;
            }
          float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float m_new = fmaxf(m_run[k], mx);
          if (m_new != -INFINITY) {
            l_run[k] = l_run[k] * exp2f(m_run[k] - m_new) + (exp2f(x[0] - m_new) + exp2f(x[1] - m_new)) +
                       (exp2f(x[2] - m_new) + exp2f(x[3] - m_new));
            m_run[k] = m_new;
          }
        }
      } else {
        // weights of prefix keys, summed over this lane's 4 rows, then over the warp's rows
        float v[4];  // keys: nt * 2 + e
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (rowok[k]) sum += exp2f(acc[k >> 1][nt][(k & 1) * 2 + e] * P.scale_log2 - Mr[k]) * Ir[k];
            v[nt * 2 + e] = sum;
          }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[j] += __shfl_xor_sync(0xffffffffu, v[j], 4);
          v[j] += __shfl_xor_sync(0xffffffffu, v[j], 8);
          v[j] += __shfl_xor_sync(0xffffffffu, v[j], 16);
        }
        if (g == 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) atomicAdd(&vacc[s * 16 + 8 * (j >> 1) + 2 * qd + (j & 1)], v[j]);
        }
      }
    }
    if (kPass == 2) {
      // the last warp to finish this page publishes its 16 votes and resets the slot
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&vcnt[s], 1) == kSnWarps - 1;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence_block();
        if (lane < 16) {
          const int key = key0 + lane;
          const float val = atomicExch(&vacc[s * 16 + lane], 0.f);
          if (key < Pfx) vrow[key] = val;
        }
        if (lane == 0) vcnt[s] = 0;
        __threadfence_block();
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
  }

  if (kPass == 1 && active) {
    float* st = P.stats + (size_t(pair) * P.chunks + chunk) * P.rows * 2;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float l = l_run[k];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (qd == 0 && rowok[k]) {
        st[rowid[k] * 2] = m_run[k];
        st[rowid[k] * 2 + 1] = l;
      }
    }
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
constexpr size_t kSnSmem = size_t(kSnStages) * kSnStageBytes + 1024 + 2 * kSnStages * 8 +
                           kSnStages * 16 * 4 + kSnStages * 4 + kSnMaxRows * 2 * 4;
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
int sn_chunks(int L, int Hkv, int S) {
  const int pages = (S + kSnPage - 1) / kSnPage;
  const int slots = sm_count();
  int c = std::max(1, (3 * slots + L * Hkv - 1) / (L * Hkv));
  c = std::min(c, std::max(1, pages / 16));
  return std::min(c, kSnMaxChunks);
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
    cudaError_t e0 = smem_limit_once(reinterpret_cast<const void*>(snap_qk_kernel<1>), int(kSnSmem));
    if (e0 == cudaSuccess) e0 = smem_limit_once(reinterpret_cast<const void*>(snap_qk_kernel<2>), int(kSnSmem));
    if (e0 == cudaSuccess)
      e0 = smem_limit_once(reinterpret_cast<const void*>(snap_select_kernel), int(sizeof(RowTopkSmem)));
    if (e0 != cudaSuccess) return cuda_fail(e0, "kvsel_snapkv_select (attribute)");
  }
  const dim3 grid(chunks, num_layers * Hkv);
  cudaError_t e;
  trace_before("snap_stats", st);
  snap_qk_kernel<1><<<grid, kSnThreads, kSnSmem, st>>>(tmK, P);
  e = cudaGetLastError();
  trace_after(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_snapkv_select (stats launch)");
  if (seq_len > obs_window) {
    trace_before("snap_vote", st);
    snap_qk_kernel<2><<<grid, kSnThreads, kSnSmem, st>>>(tmK, P);
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
