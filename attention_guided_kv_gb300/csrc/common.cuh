// Shared device/host helpers for the kvsel kernels (sm_103a).
//
// Device side: thin inline-PTX wrappers for mbarriers, TMA tensor loads,
// ldmatrix and the bf16 mma.sync used by the decode kernels, plus the
// device status word every kernel reports problems into.
// Host side: the per-thread error string, argument-check helpers and the
// tensor-map encoder (fetched from the driver at run time, no -lcuda).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/kvsel.h"

namespace kvsel {

// ---------------------------------------------------------------------------
// device status word: first bytes of every workspace
// ---------------------------------------------------------------------------
constexpr size_t kStatusBytes = 256;

// Pool pages hold 16, 32, 64, 128 or 256 tokens; kernels address them in
// 16-token tiles.  Returns log2(page_size / 16), or -1 for any other size.
__host__ __device__ inline int page_shift_of(int page_size) {
  for (int s = 0; s <= 4; ++s)
    if (page_size == (16 << s)) return s;
  return -1;
}

__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Waits on other CTAs (a readiness counter, a grid barrier) spin a bounded
// number of times, each spin a short sleep.  The bound is the kernel's
// default (a few seconds) unless the workspace's status block holds a
// non-zero override at this byte offset (kvsel_set_wait_limit).
constexpr size_t kWaitLimitOffset = 32;
__device__ __forceinline__ unsigned spin_limit(const int* status, unsigned dflt) {
  if (!status) return dflt;
  const unsigned v =
      __ldcg(reinterpret_cast<const unsigned*>(reinterpret_cast<const uint8_t*>(status) + kWaitLimitOffset));
  return v ? v : dflt;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier (CTA scope)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: every try_wait suspends for at most a short hardware-defined
// interval, so 2^22 attempts bound the wait at a few seconds.  On expiry the
// status word gets KVSEL_ERR_TIMEOUT and the caller stops using the stage.
constexpr uint32_t kWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status) {
#pragma unroll 1
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  report(status, KVSEL_ERR_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2D tiled load of one box into shared memory, completing on `bar`.
// x (innermost coordinate) must make x * elem_size a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// 3D tiled load (see encode_bf16_row_pages): one instruction moves a whole
// box of rows x 128 bf16 as two 64-column halves, 128-byte swizzled.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}
// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
// Order this thread's earlier generic-proxy global writes before later
// async-proxy (TMA) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------------------
// warp-level matrix ops
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Monotone map fp32 -> uint32 (a < b as floats <=> key(a) < key(b)); -0 maps like +0.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace kvsel

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
namespace kvsel_host {

void set_error(const std::string& msg);
kvsel_status fail(kvsel_status code, const std::string& msg);
kvsel_status cuda_fail(cudaError_t err, const char* what);
bool aligned(const void* p, size_t a);
int sm_count();
// Raise a kernel's dynamic shared memory limit to `bytes`, once per device.
cudaError_t smem_limit_once(const void* fn, int bytes);
// Encode a 2D bf16 tensor map with 128-byte swizzle over a [rows][inner] array.
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);
// The same [rows][128] bf16 array as a 3D tensor {64 columns, rows, 2 halves}
// (strides 256 B and 128 B) with boxes of {64, box_rows, 2}: one TMA load puts
// box_rows whole rows in shared memory as two [box_rows][128 B] halves, the
// second 64 * box_rows * 2 bytes after the first -- the layout two 2D loads of
// 64-column boxes would write, at half the instructions.
bool encode_bf16_row_pages(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
// Launch tracing (see kvsel_trace_start): call around every kernel launch.
void trace_before(const char* kernel, cudaStream_t st);
void trace_after(cudaStream_t st);

}  // namespace kvsel_host
