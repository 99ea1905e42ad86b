// sp24_internal.cuh -- host-side helpers shared by the library's translation
// units: per-device state (SM count, architecture check, the device error
// word), tensor-map encoding through the driver entry point, and argument
// checks.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>
#include "../../include/sp24.h"

namespace sp24 {

// Device error word bits, set by kernels with atomicOr.
enum : unsigned int {
  DEVERR_TIMEOUT_PRODUCER = 1u,
  DEVERR_TIMEOUT_MMA = 2u,
  DEVERR_TIMEOUT_EPILOGUE = 4u,
};

struct DeviceInfo {
  int ordinal = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
  unsigned int* err_word = nullptr;  // device address of the error word
};

// Current device's info (created on first use).  Returns SP24_ERR_CUDA or
// SP24_ERR_ARCH on failure.
sp24_status current_device(const DeviceInfo** out);

// 2D tensor map over a row-major [rows][cols] array of `elem_bytes`-sized
// elements with row stride `row_stride_bytes`; box {box_cols, box_rows};
// out-of-range elements read as zero.
// 3D: [depth][rows][cols] with row and depth strides in bytes (a batch of 2D views).
sp24_status make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                         uint64_t depth, uint64_t row_stride_bytes, uint64_t depth_stride_bytes, uint32_t box_cols,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle);
sp24_status make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols,
                         uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swizzle);

// Launches `kern` with programmatic stream serialisation: it may begin while
// the previous kernel in the stream finishes, and must call pdl_wait() (see
// sp24_ptx.cuh) before its first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace sp24
