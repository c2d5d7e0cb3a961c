// Host-side plumbing shared by every entry point: the per-thread error
// string, the workspace status word, the tensor-map encoder and the launch
// trace (CUDA events for the bench, NVTX ranges for a timeline profiler).
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdlib>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "common.cuh"

namespace kvsel_host {

static thread_local std::string g_error;

void set_error(const std::string& msg) { g_error = msg; }

kvsel_status fail(kvsel_status code, const std::string& msg) {
  g_error = msg;
  return code;
}

kvsel_status cuda_fail(cudaError_t err, const char* what) {
  g_error = std::string(what) + ": " + cudaGetErrorString(err);
  return KVSEL_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

cudaError_t smem_limit_once(const void* fn, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, fn})) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({dev, fn});
  return e;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_bf16_row_pages(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, 2};
  cuuint64_t strides[2] = {256, 128};  // bytes: next row, next 64-column half
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct TraceState {
  void* const* events = nullptr;
  int capacity = 0;
  int count = 0;
  std::vector<const char*> names;
};
static thread_local TraceState g_trace;

// NVTX ranges around every library launch (named after the kernel) for a
// timeline profiler, when the environment sets KVSEL_NVTX=1; read once.
static bool nvtx_on() {
  static const bool on = [] {
    const char* v = std::getenv("KVSEL_NVTX");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

void trace_before(const char* kernel, cudaStream_t st) {
  if (nvtx_on()) nvtxRangePushA(kernel);
  TraceState& t = g_trace;
  if (!t.events || t.count >= t.capacity) return;
  t.names.push_back(kernel);
  cudaEventRecord(static_cast<cudaEvent_t>(t.events[2 * t.count]), st);
}

void trace_after(cudaStream_t st) {
  if (nvtx_on()) nvtxRangePop();
  TraceState& t = g_trace;
  if (!t.events || t.count >= t.capacity) return;
  cudaEventRecord(static_cast<cudaEvent_t>(t.events[2 * t.count + 1]), st);
  ++t.count;
}

}  // namespace kvsel_host

using namespace kvsel_host;

extern "C" kvsel_status kvsel_trace_start(void* const* events, int capacity) {
  if (!events || capacity < 1) return fail(KVSEL_ERR_INVALID_ARG, "kvsel_trace_start: need events and capacity >= 1");
  g_trace.events = events;
  g_trace.capacity = capacity;
  g_trace.count = 0;
  g_trace.names.clear();
  g_trace.names.reserve(size_t(capacity));
  return KVSEL_OK;
}

extern "C" int kvsel_trace_stop(const char** names, int capacity) {
  const int n = g_trace.count;
  if (names)
    for (int i = 0; i < n && i < capacity; ++i) names[i] = g_trace.names[size_t(i)];
  g_trace.events = nullptr;
  g_trace.capacity = 0;
  g_trace.count = 0;
  return n;
}

extern "C" const char* kvsel_last_error_string(void) { return g_error.c_str(); }

extern "C" kvsel_status kvsel_clear_status(void* workspace, void* stream) {
  if (!workspace) return fail(KVSEL_ERR_INVALID_ARG, "kvsel_clear_status: workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_clear_status");
  return KVSEL_OK;
}

namespace {
__global__ void set_wait_limit_kernel(unsigned* word, unsigned spins) { *word = spins; }
}  // namespace

extern "C" kvsel_status kvsel_set_wait_limit(void* workspace, unsigned spins, void* stream) {
  if (!workspace || !aligned(workspace, 256))
    return fail(KVSEL_ERR_INVALID_ARG, "kvsel_set_wait_limit: a 256-byte aligned workspace is required");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  set_wait_limit_kernel<<<1, 1, 0, st>>>(
      reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + kvsel::kWaitLimitOffset), spins);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return cuda_fail(e, "kvsel_set_wait_limit");
  return KVSEL_OK;
}

extern "C" kvsel_status kvsel_read_status(void* workspace, void* stream) {
  if (!workspace) return fail(KVSEL_ERR_INVALID_ARG, "kvsel_read_status: workspace is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int code = 0;
  cudaError_t e = cudaMemcpyAsync(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "kvsel_read_status");
  if (code != 0) {
    e = cudaMemsetAsync(workspace, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "kvsel_read_status (clear)");
    set_error(code == KVSEL_ERR_TIMEOUT     ? "device: a bounded wait ran out"
              : code == KVSEL_ERR_BAD_INDEX ? "device: block-table entry outside the page pool"
                                            : "device: error");
  }
  return static_cast<kvsel_status>(code);
}
