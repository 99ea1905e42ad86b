// sp24_abi.cu -- status strings, per-device state, the device error word,
// tensor-map encoding, and sp24_last_device_error.
#include <mutex>
#include "sp24_internal.cuh"

namespace sp24 {

// One word per device: kernels OR error bits into it when a bounded wait
// gives up; sp24_last_device_error reads and clears it.
__device__ unsigned int g_device_error_word;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
bool g_ready[kMaxDevices] = {};
std::mutex g_mutex;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
}  // namespace

sp24_status current_device(const DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SP24_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_ready[dev]) {
    DeviceInfo d;
    d.ordinal = dev;
    int smem = 0;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return SP24_ERR_CUDA;
    d.smem_optin = static_cast<size_t>(smem);
    if (d.cc_major != 10 || d.cc_minor != 3) return SP24_ERR_ARCH;  // kernels are built for sm_103a only
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err_word), g_device_error_word) != cudaSuccess)
      return SP24_ERR_CUDA;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return SP24_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    g_devices[dev] = d;
    g_ready[dev] = true;
  }
  *out = &g_devices[dev];
  return SP24_OK;
}

sp24_status make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols,
                         uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swizzle) {
  if (!g_encode) return SP24_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SP24_OK : SP24_ERR_CUDA;
}

sp24_status make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                         uint64_t depth, uint64_t row_stride_bytes, uint64_t depth_stride_bytes, uint32_t box_cols,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  if (!g_encode) return SP24_ERR_CUDA;
  cuuint64_t dims[3] = {cols, rows, depth};
  cuuint64_t strides[2] = {row_stride_bytes, depth_stride_bytes};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SP24_OK : SP24_ERR_CUDA;
}

}  // namespace sp24

extern "C" {

const char* sp24_status_string(sp24_status s) {
  switch (s) {
    case SP24_OK: return "SP24_OK";
    case SP24_ERR_INVALID_ARG: return "SP24_ERR_INVALID_ARG: null pointer, bad size or stride";
    case SP24_ERR_UNSUPPORTED: return "SP24_ERR_UNSUPPORTED: valid but not implemented";
    case SP24_ERR_ALIGNMENT: return "SP24_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
    case SP24_ERR_CUDA: return "SP24_ERR_CUDA: a CUDA call failed";
    case SP24_ERR_ARCH: return "SP24_ERR_ARCH: device is not sm_103";
    case SP24_ERR_WORKSPACE: return "SP24_ERR_WORKSPACE: workspace missing or too small";
    case SP24_ERR_DEVICE_TIMEOUT: return "SP24_ERR_DEVICE_TIMEOUT: a kernel gave up on a bounded wait";
  }
  return "SP24_ERR_UNKNOWN";
}

size_t sp24_meta_bytes(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0 || K % 8 != 0) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K / 8);
}

sp24_status sp24_last_device_error(void* stream) {
  const sp24::DeviceInfo* dev = nullptr;
  sp24_status st = sp24::current_device(&dev);
  if (st != SP24_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SP24_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, dev->err_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return SP24_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(dev->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return SP24_ERR_CUDA;
    return SP24_ERR_DEVICE_TIMEOUT;
  }
  return SP24_OK;
}

}  // extern "C"
