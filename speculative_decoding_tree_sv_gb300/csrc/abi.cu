// Host-side common entry points: version, status names, the device error
// word, driver entry-point resolution for tensor maps, SM count; and a
// self-test of the bounded device wait.
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
std::mutex g_sm_mutex;
}  // namespace

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                      CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  });
  if (g_encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  return g_encode(map, dtype, rank, base, dims, strides_bytes, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_sm_mutex);
    if (g_sm_count[dev] > 0) return g_sm_count[dev];
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  if (dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_sm_mutex);
    g_sm_count[dev] = n;
  }
  return n;
}

// A wait that can never complete: one CTA initialises an mbarrier that
// nothing arrives on and waits for its first phase with the bounded wait
// every kernel of the library uses.  With `abort_after_ns` > 0 a second warp
// raises the shared abort flag after that long instead, the way a role of a
// kernel stops the others.  Either way the wait gives up, SV_DEVERR_TIMEOUT
// is recorded and the kernel returns normally.
__global__ void __launch_bounds__(64) bounded_wait_selftest_kernel(int* err, unsigned long long abort_after_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, &abort_flag)) report_error(err, SV_DEVERR_TIMEOUT);
  } else if (threadIdx.x == 32 && abort_after_ns > 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < abort_after_ns) {
    }
    *reinterpret_cast<volatile int*>(&abort_flag) = 1;
  }
}

}  // namespace sv

extern "C" {

int sv_abi_version(void) { return 2; }

sv_status sv_selftest_bounded_wait(void* workspace, long long abort_after_ns, sv_stream_t stream) {
  if (workspace == nullptr || abort_after_ns < 0 || abort_after_ns >= static_cast<long long>(sv::kWaitTimeoutNs))
    return SV_ERR_INVALID_ARG;
  sv::bounded_wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(workspace), static_cast<unsigned long long>(abort_after_ns));
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

const char* sv_status_string(sv_status status) {
  switch (status) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: null pointer, bad size or misaligned pointer";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: shape outside the supported set";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA call or kernel launch failed";
    case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing or too small";
    case SV_ERR_DEVICE: return "SV_ERR_DEVICE: a kernel reported a device error code";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded device wait ran out";
  }
  return "unknown sv_status";
}

sv_status sv_get_device_error(void* workspace, int* code, sv_stream_t stream) {
  if (workspace == nullptr || code == nullptr) return SV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int value = 0;
  if (cudaMemcpyAsync(&value, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  *code = value;
  if (value != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
    return value == SV_DEVERR_TIMEOUT ? SV_ERR_TIMEOUT : SV_ERR_DEVICE;
  }
  return SV_OK;
}

}  // extern "C"
