// Host-side common entry points: version, status names, the device error
// word, driver entry-point resolution for tensor maps, SM count.
#include <mutex>

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

}  // namespace sv

extern "C" {

int sv_abi_version(void) { return 2; }

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
