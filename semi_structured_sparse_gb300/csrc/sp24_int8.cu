// sp24_int8.cu -- the int8 x int8 2:4 sparse GEMM, the int8 sibling of the
// FP8 path (pytorch/ao PR #3258, review: the 2:4 kernels are int8 x int8 and
// fp8 x fp8; Int8SemiSparseTensor):
//
//   Y[m][n] = bf16( (sx[m] sw[n]) * float(acc[m][n]) + bias[n] ),
//   acc[m][n] = sum over the kept k of wq[n][k] xq[m][k]   (exact, int32)
//
// with per-token activation scales and per-channel weight scales.  The
// weight is the FP8 path's storage with int8 codes (sp24_int8_compress): the
// same tiled values and metadata.
//
// sm_103a has no int8 tcgen05 MMA (kind::i8 is not available on this target),
// so this kernel runs on the legacy warp-level sparse MMA,
// mma.sp::ordered_metadata m16n8k64 s8 x s8 -> s32.  Its register layouts
// (measured on the GPU with one-hot operands): for lane l, g = l / 4 and
// t = l % 4,
//   A  a0 / a1: row g / g + 8, kept bytes 4t .. 4t + 3 of the 32 kept of the
//      16 x 64 slice; a2 / a3: the same rows, kept bytes 16 + 4t .. + 3;
//   B  b_R: column (token) g, k = 16 R + 4t .. + 3;
//   metadata: row g + 8 (t % 2), the 4-bit groups 8 (t / 2) .. + 7 of the
//      row's slice, in the storage's logical nibble order -- one 32-bit
//      word of the tiled metadata;
//   D  d0, d1: row g, columns 2t, 2t + 1; d2, d3: row g + 8.
// So every operand word is one aligned 32-bit load from the weight storage
// or the activation rows; no shared memory.  A CTA of 4 warps computes 64
// weight rows x 64 tokens; each warp 32 x 32 (2 x 4 MMAs per 64-wide K slice).
#include <cuda_bf16.h>
#include "sp24_internal.cuh"
#include "sp24_ptx.cuh"

namespace sp24 {
namespace {

constexpr int kI8Rows = 64;    // weight rows per CTA
constexpr int kI8Tokens = 64;  // tokens per CTA

__device__ __forceinline__ void mma_sp_s8(int (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[4], uint32_t e) {
  asm volatile(
      "mma.sp::ordered_metadata.sync.aligned.m16n8k64.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, 0x0;"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(e));
}

__global__ void __launch_bounds__(128) sp24_int8_gemm_kernel(const uint8_t* __restrict__ Xq, const float* __restrict__ sx,
                                                             int M, int K, int64_t ldx, const uint8_t* __restrict__ values,
                                                             const uint8_t* __restrict__ meta,
                                                             const float* __restrict__ sw, int N,
                                                             const uint16_t* __restrict__ bias,
                                                             uint16_t* __restrict__ Y, int64_t ldy) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n_base = blockIdx.y * kI8Rows + 32 * (warp >> 1);   // this warp's 32 weight rows
  const int m_base = blockIdx.x * kI8Tokens + 32 * (warp & 1);  // this warp's 32 tokens
  const int ktiles = K >> 7;
  pdl_wait();
  // per row block (16 rows): the thread's A rows g, g + 8 and metadata row g + 8 (t % 2)
  const uint8_t* arow[2][2];
  const uint8_t* mrow[2];
  int aswz[2][2];
  for (int rb = 0; rb < 2; ++rb) {
    for (int hh = 0; hh < 2; ++hh) {
      const int n = n_base + 16 * rb + g + 8 * hh;
      arow[rb][hh] = values + static_cast<int64_t>(n >> 7) * ktiles * 8192 + (n & 127) * 64 + 4 * t;
      aswz[rb][hh] = ((n & 127) >> 1) & 3;
    }
    const int nm = n_base + 16 * rb + g + 8 * (t & 1);
    mrow[rb] = meta + static_cast<int64_t>(nm >> 7) * ktiles * 2048 + (nm & 127) * 16 + 4 * (t >> 1);
  }
  // per token block (8 tokens): the thread's token row (clamped to M - 1; its results are not stored)
  const uint8_t* xrow[4];
  for (int tb = 0; tb < 4; ++tb) {
    const int m = min(m_base + 8 * tb + g, M - 1);
    xrow[tb] = Xq + static_cast<int64_t>(m) * ldx + 4 * t;
  }
  int acc[2][4][4];
#pragma unroll
  for (int rb = 0; rb < 2; ++rb)
#pragma unroll
    for (int tb = 0; tb < 4; ++tb)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[rb][tb][i] = 0;
  for (int ks = 0; ks < (K >> 6); ++ks) {
    const int tile = ks >> 1, sub = ks & 1;
    uint32_t a[2][4], e[2], b[4][4];
#pragma unroll
    for (int rb = 0; rb < 2; ++rb) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // a0..a3: (row half q % 2, kept bytes 16 (q / 2) + 4t)
        const int hh = q & 1, chunk = 2 * sub + (q >> 1);
        a[rb][q] = __ldg(reinterpret_cast<const uint32_t*>(arow[rb][hh] + static_cast<int64_t>(tile) * 8192 +
                                                           ((chunk ^ aswz[rb][hh]) << 4)));
      }
      e[rb] = __ldg(reinterpret_cast<const uint32_t*>(mrow[rb] + static_cast<int64_t>(tile) * 2048 + 8 * sub));
    }
#pragma unroll
    for (int tb = 0; tb < 4; ++tb)
#pragma unroll
      for (int R = 0; R < 4; ++R)
        b[tb][R] = __ldg(reinterpret_cast<const uint32_t*>(xrow[tb] + 64 * ks + 16 * R));
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
      for (int tb = 0; tb < 4; ++tb) mma_sp_s8(acc[rb][tb], a[rb], b[tb], e[rb]);
  }
  // epilogue: y = (sx sw) * float(acc) (+ bias), each step rounded as written, then bf16
#pragma unroll
  for (int rb = 0; rb < 2; ++rb)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n = n_base + 16 * rb + g + 8 * hh;
      const float swn = __ldg(&sw[n]);
      const float bn = bias ? __uint_as_float(static_cast<uint32_t>(__ldg(&bias[n])) << 16) : 0.0f;
#pragma unroll
      for (int tb = 0; tb < 4; ++tb)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int m = m_base + 8 * tb + 2 * t + c;
          if (m < M) {
            float y = __fmul_rn(__fmul_rn(__ldg(&sx[m]), swn), __int2float_rn(acc[rb][tb][2 * hh + c]));
            if (bias) y = __fadd_rn(y, bn);
            Y[static_cast<int64_t>(m) * ldy + n] = static_cast<uint16_t>(bf16x2_rn(y, 0.0f) & 0xFFFFu);
          }
        }
    }
  pdl_trigger();
}

}  // namespace
}  // namespace sp24

extern "C" sp24_status sp24_int8_gemm(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx,
                                      const void* values, const void* meta, const float* sw, int64_t N,
                                      const void* bias, void* Y, int64_t ldy, void* stream) {
  using namespace sp24;
  if (!Xq || !sx || !values || !meta || !sw || !Y) return SP24_ERR_INVALID_ARG;
  if (M < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0) return SP24_ERR_INVALID_ARG;
  if (M > (1 << 30) || N > (1 << 30)) return SP24_ERR_INVALID_ARG;
  if (K > 131072) return SP24_ERR_UNSUPPORTED;  // the int32 sums stay exact: K/2 * 127^2 < 2^31
  if (ldx < K || ldy < N) return SP24_ERR_INVALID_ARG;
  if (!aligned16(Xq) || !aligned16(values) || !aligned16(meta) || ldx % 16 != 0) return SP24_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(sx) | reinterpret_cast<uintptr_t>(sw)) % 4 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(Y) % 2 != 0 || reinterpret_cast<uintptr_t>(bias) % 2 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  const sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;
  const dim3 grid(static_cast<unsigned>((M + kI8Tokens - 1) / kI8Tokens), static_cast<unsigned>(N / kI8Rows));
  if (grid.y > 65535u) return SP24_ERR_UNSUPPORTED;
  if (launch_pdl(sp24_int8_gemm_kernel, grid, dim3(128), 0, static_cast<cudaStream_t>(stream),
                 static_cast<const uint8_t*>(Xq), sx, (int)M, (int)K, ldx, static_cast<const uint8_t*>(values),
                 static_cast<const uint8_t*>(meta), sw, (int)N, static_cast<const uint16_t*>(bias),
                 static_cast<uint16_t*>(Y), ldy) != cudaSuccess)
    return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}
