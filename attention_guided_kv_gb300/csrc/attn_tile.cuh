// One 16-key attention tile for the GQA decode kernels (sm_103a, mma.sync).
//
// A tile holds 16 keys of one kv head in shared memory: K and V each as two
// 64-column halves of 16 rows x 128 bytes, with the 128-byte swizzle (16-byte
// unit u of row r stored at unit u ^ (r & 7)), the layout a TMA box with
// CU_TENSOR_MAP_SWIZZLE_128B produces and the gather kernels reproduce.
//
// The group's q rows are the A operand of S = Q K^T.  Up to 8 heads (rows
// 8..15 zero), P is split into bf16(p) (A rows 0..7) and bf16(p - bf16(p))
// (rows 8..15) for O += P V, so the probabilities keep ~16 mantissa bits at
// no extra MMA.  With 9..16 heads (attend_tile_wide), head g + 8 takes rows
// g + 8 and a second MMA adds the residuals.  Each lane of a warp owns head
// g = lane / 4 (and g + 8) and keys {2q, 2q+1, 8+2q, 9+2q} (q = lane % 4) of
// the tile.
#pragma once

#include "common.cuh"

namespace kvsel {

__device__ __forceinline__ uint32_t tile_unit_off(int key, int u) {
  return (u >> 3) * 2048 + key * 128 + ((((u & 7) ^ (key & 7))) << 4);
}
__device__ __forceinline__ uint32_t tile_keep_keys(uint32_t v, int k0, int valid) {
  return v & ((k0 < valid ? 0x0000FFFFu : 0u) | (k0 + 1 < valid ? 0xFFFF0000u : 0u));
}

struct TileState {
  float m = -INFINITY, l = 0.f;    // running max (log2 domain) and this lane's partial sum, head g
  float m2 = -INFINITY, l2 = 0.f;  // head g + 8 (attend_tile_wide)
  float o[16][4];                  // O accumulators: [n-tile of 8 dims][row g pair, row g + 8 pair]
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }
};

// Load the A fragments of the group's q rows: qa[kt][0..1] for k-tile kt.
__device__ __forceinline__ void load_q_frags(const __nv_bfloat16* qrow, bool head_ok, int qd,
                                             uint32_t (&qa)[8][2]) {
  const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
    qa[kt][0] = head_ok ? q32[(16 * kt + 2 * qd) >> 1] : 0u;
    qa[kt][1] = head_ok ? q32[(16 * kt + 8 + 2 * qd) >> 1] : 0u;
  }
}

// Process one tile of `valid` (1..16) keys at shared addresses kb / vb.
// Returns the lane's four scaled log2 logits (-inf for keys >= valid).  A
// lane whose head is off for this tile (head_on false) sees every logit as
// -inf; its state is unchanged, also while it has seen no key yet.
__device__ __forceinline__ void attend_tile(uint32_t kb, uint32_t vb, const uint32_t (&qa)[8][2],
                                            int valid, float scale_log2, TileState& st, float& x0,
                                            float& x1, float& x2, float& x3, bool head_on = true) {
  const int lane = threadIdx.x & 31, qd = lane & 3, mi = lane >> 3, r8 = lane & 7;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
    const int key = (mi >> 1) * 8 + r8;
    const int uu = 2 * kt + (mi & 1);
    uint32_t b0, b1, b2, b3;
    ldsm_x4(kb + tile_unit_off(key, uu), b0, b1, b2, b3);
    mma_bf16_16816(s0, qa[kt][0], 0u, qa[kt][1], 0u, b0, b1);
    mma_bf16_16816(s1, qa[kt][0], 0u, qa[kt][1], 0u, b2, b3);
  }
  const int k0 = 2 * qd, k2 = 8 + 2 * qd;
  x0 = head_on && k0 < valid ? s0[0] * scale_log2 : -INFINITY;
  x1 = head_on && k0 + 1 < valid ? s0[1] * scale_log2 : -INFINITY;
  x2 = head_on && k2 < valid ? s1[0] * scale_log2 : -INFINITY;
  x3 = head_on && k2 + 1 < valid ? s1[1] * scale_log2 : -INFINITY;
  float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(st.m, mx);
  const float m_ref = m_new == -INFINITY ? 0.f : m_new;  // nothing seen yet: alpha and p come out 0
  const float alpha = exp2f(st.m - m_ref);
  const float p0 = exp2f(x0 - m_ref), p1 = exp2f(x1 - m_ref);
  const float p2 = exp2f(x2 - m_ref), p3 = exp2f(x3 - m_ref);
  st.l = st.l * alpha + ((p0 + p1) + (p2 + p3));
  st.m = m_new;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    st.o[nt][0] *= alpha;
    st.o[nt][1] *= alpha;
    st.o[nt][2] *= alpha;
    st.o[nt][3] *= alpha;
  }
  const uint32_t hi01 = pack_bf16x2(p0, p1);
  const uint32_t hi23 = pack_bf16x2(p2, p3);
  const uint32_t lo01 = pack_bf16x2(p0 - bf16lo_to_f32(hi01), p1 - bf16hi_to_f32(hi01));
  const uint32_t lo23 = pack_bf16x2(p2 - bf16lo_to_f32(hi23), p3 - bf16hi_to_f32(hi23));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int key = (mi & 1) * 8 + r8;
    const int uu = 2 * j + (mi >> 1);
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vb + tile_unit_off(key, uu), b0, b1, b2, b3);
    if (valid < 16) {  // rows past the valid keys may hold anything
      b0 = tile_keep_keys(b0, 2 * qd, valid);
      b1 = tile_keep_keys(b1, 8 + 2 * qd, valid);
      b2 = tile_keep_keys(b2, 2 * qd, valid);
      b3 = tile_keep_keys(b3, 8 + 2 * qd, valid);
    }
    mma_bf16_16816(st.o[2 * j], hi01, lo01, hi23, lo23, b0, b1);
    mma_bf16_16816(st.o[2 * j + 1], hi01, lo01, hi23, lo23, b2, b3);
  }
}

// The same for a group of 9..16 heads: qb holds head g + 8's A fragments (zero
// for lanes whose g + 8 is past the group); on / on2 switch heads g / g + 8
// off for this tile as attend_tile's head_on does.
__device__ __forceinline__ void attend_tile_wide(uint32_t kb, uint32_t vb, const uint32_t (&qa)[8][2],
                                                 const uint32_t (&qb)[8][2], int valid, float scale_log2,
                                                 TileState& st, bool on, bool on2) {
  const int lane = threadIdx.x & 31, qd = lane & 3, mi = lane >> 3, r8 = lane & 7;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
    const int key = (mi >> 1) * 8 + r8;
    const int uu = 2 * kt + (mi & 1);
    uint32_t b0, b1, b2, b3;
    ldsm_x4(kb + tile_unit_off(key, uu), b0, b1, b2, b3);
    mma_bf16_16816(s0, qa[kt][0], qb[kt][0], qa[kt][1], qb[kt][1], b0, b1);
    mma_bf16_16816(s1, qa[kt][0], qb[kt][0], qa[kt][1], qb[kt][1], b2, b3);
  }
  const int k0 = 2 * qd, k2 = 8 + 2 * qd;
  // one head's four logits -> its probabilities, with the running (max, sum) and the rescale of
  // its O row pair (c = 0: row g, c = 2: row g + 8)
  auto head = [&](float a, float bb, float cc, float dd, bool hon, float& m, float& l, int c, float (&p)[4]) {
    const float x0 = hon && k0 < valid ? a * scale_log2 : -INFINITY;
    const float x1 = hon && k0 + 1 < valid ? bb * scale_log2 : -INFINITY;
    const float x2 = hon && k2 < valid ? cc * scale_log2 : -INFINITY;
    const float x3 = hon && k2 + 1 < valid ? dd * scale_log2 : -INFINITY;
    float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float m_ref = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2f(m - m_ref);
    p[0] = exp2f(x0 - m_ref);
    p[1] = exp2f(x1 - m_ref);
    p[2] = exp2f(x2 - m_ref);
    p[3] = exp2f(x3 - m_ref);
    l = l * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
    m = m_new;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      st.o[nt][c] *= alpha;
      st.o[nt][c + 1] *= alpha;
    }
  };
  float pa[4], pb[4];
  head(s0[0], s0[1], s1[0], s1[1], on, st.m, st.l, 0, pa);
  head(s0[2], s0[3], s1[2], s1[3], on2, st.m2, st.l2, 2, pb);
  const uint32_t hiA = pack_bf16x2(pa[0], pa[1]), hiC = pack_bf16x2(pa[2], pa[3]);
  const uint32_t hiB = pack_bf16x2(pb[0], pb[1]), hiD = pack_bf16x2(pb[2], pb[3]);
  const uint32_t loA = pack_bf16x2(pa[0] - bf16lo_to_f32(hiA), pa[1] - bf16hi_to_f32(hiA));
  const uint32_t loC = pack_bf16x2(pa[2] - bf16lo_to_f32(hiC), pa[3] - bf16hi_to_f32(hiC));
  const uint32_t loB = pack_bf16x2(pb[0] - bf16lo_to_f32(hiB), pb[1] - bf16hi_to_f32(hiB));
  const uint32_t loD = pack_bf16x2(pb[2] - bf16lo_to_f32(hiD), pb[3] - bf16hi_to_f32(hiD));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int key = (mi & 1) * 8 + r8;
    const int uu = 2 * j + (mi >> 1);
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vb + tile_unit_off(key, uu), b0, b1, b2, b3);
    if (valid < 16) {
      b0 = tile_keep_keys(b0, 2 * qd, valid);
      b1 = tile_keep_keys(b1, 8 + 2 * qd, valid);
      b2 = tile_keep_keys(b2, 2 * qd, valid);
      b3 = tile_keep_keys(b3, 8 + 2 * qd, valid);
    }
    mma_bf16_16816(st.o[2 * j], hiA, hiB, hiC, hiD, b0, b1);
    mma_bf16_16816(st.o[2 * j + 1], hiA, hiB, hiC, hiD, b2, b3);
    mma_bf16_16816(st.o[2 * j], loA, loB, loC, loD, b0, b1);
    mma_bf16_16816(st.o[2 * j + 1], loA, loB, loC, loD, b2, b3);
  }
}

// ---------------------------------------------------------------------------
// Split-KV partial results of one (sequence, kv head): a slot per split holds
// every head's running max M (log2 domain), sum L and unnormalised O.
constexpr int kTileMaxG = 16;
constexpr int kTileD = 128;
constexpr int kTileMaxSplits = 64;
constexpr int kPartFloats = kTileMaxG * (kTileD + 2);  // [M x 16][L x 16][O 16 x 128]

// Merge the kWarps warps' tile states of one CTA into its split slot.  wo:
// shared scratch of kWarps x kTileMaxG x (kTileD + 2) floats.  Every thread
// of the CTA calls it (it synchronises the block).  kWide: the states come
// from attend_tile_wide (rows g + 8 are head g + 8, not residuals).
template <int kWarps, bool kWide = false>
__device__ __forceinline__ void merge_warps_to_slot(const TileState& st, float* wo, float* slot, int G) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, qd = lane & 3;
  float l = st.l, l2 = st.l2;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  l2 += __shfl_xor_sync(0xffffffffu, l2, 1);
  l2 += __shfl_xor_sync(0xffffffffu, l2, 2);
  float* mine = wo + (warp * kTileMaxG + g) * (kTileD + 2);
  if (g < G) {
    if (qd == 0) {
      mine[kTileD] = st.m;
      mine[kTileD + 1] = l;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      mine[8 * nt + 2 * qd] = kWide ? st.o[nt][0] : st.o[nt][0] + st.o[nt][2];
      mine[8 * nt + 2 * qd + 1] = kWide ? st.o[nt][1] : st.o[nt][1] + st.o[nt][3];
    }
  }
  if (kWide && g + 8 < G) {
    float* mine2 = wo + (warp * kTileMaxG + g + 8) * (kTileD + 2);
    if (qd == 0) {
      mine2[kTileD] = st.m2;
      mine2[kTileD + 1] = l2;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      mine2[8 * nt + 2 * qd] = st.o[nt][2];
      mine2[8 * nt + 2 * qd + 1] = st.o[nt][3];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * kTileD; idx += kWarps * 32) {
    const int gg = idx / kTileD, dd = idx % kTileD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wo[(w * kTileMaxG + gg) * (kTileD + 2) + kTileD]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* pw = wo + (w * kTileMaxG + gg) * (kTileD + 2);
        const float f = pw[kTileD] == -INFINITY ? 0.f : exp2f(pw[kTileD] - M);
        L += pw[kTileD + 1] * f;
        acc += pw[dd] * f;
      }
    }
    slot[2 * kTileMaxG + gg * kTileD + dd] = acc;
    if (dd == 0) {
      slot[gg] = M;
      slot[kTileMaxG + gg] = L;
    }
  }
}

// Merge `splits` slots (consecutive, from `part`) into the G heads' outputs
// out[(out_row0 + g) * 128 + d], fp32 or bf16.  scratch: 3 x kTileMaxSplits x
// kTileMaxG + 2 x kTileMaxG floats of shared memory.  Every thread of the CTA
// calls it.
__device__ __forceinline__ void merge_split_slots(const float* part, int splits, int G, void* out, bool out_f32,
                                                  size_t out_row0, float* scratch) {
  float (*sm)[kTileMaxG] = reinterpret_cast<float (*)[kTileMaxG]>(scratch);
  float (*sl)[kTileMaxG] = sm + kTileMaxSplits;
  float (*sf)[kTileMaxG] = sl + kTileMaxSplits;
  float* sM = &sf[kTileMaxSplits][0];
  float* sI = sM + kTileMaxG;
  for (int t = threadIdx.x; t < splits * G; t += blockDim.x) {  // every (split, head) at once
    const int sp = t / G, gg = t % G;
    const float* slot = part + size_t(sp) * kPartFloats;
    sm[sp][gg] = slot[gg];
    sl[sp][gg] = slot[kTileMaxG + gg];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int gg = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, sm[sp][gg]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int sp = 0; sp < splits; ++sp)
        if (sm[sp][gg] != -INFINITY) L += sl[sp][gg] * exp2f(sm[sp][gg] - M);
    sM[gg] = M;
    sI[gg] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  for (int t = threadIdx.x; t < splits * G; t += blockDim.x) {
    const int sp = t / G, gg = t % G;
    sf[sp][gg] = (sM[gg] != -INFINITY && sm[sp][gg] != -INFINITY) ? exp2f(sm[sp][gg] - sM[gg]) * sI[gg] : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * kTileD; idx += blockDim.x) {
    const int gg = idx / kTileD, dd = idx % kTileD;
    float acc = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < splits; ++sp) acc += sf[sp][gg] * part[size_t(sp) * kPartFloats + 2 * kTileMaxG + gg * kTileD + dd];
    const size_t oi = (out_row0 + gg) * kTileD + dd;
    if (out_f32) static_cast<float*>(out)[oi] = acc;
    else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(acc);
  }
}

}  // namespace kvsel
