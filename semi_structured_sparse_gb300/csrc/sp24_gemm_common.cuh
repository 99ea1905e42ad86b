// sp24_gemm_common.cuh -- definitions shared by the GEMM translation units
// (the one-CTA kernel in sp24_gemm.cu, the SM-pair kernel in
// sp24_gemm_pair.cu): tile constants, the kernel argument block, the epilogue
// barriers and TMEM column loads, and the pair kernel's host entry.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "sp24_internal.cuh"
#include "sp24_ptx.cuh"

namespace sp24 {

struct GemmArgs {
  const uint8_t* values;  // tiled kept values
  const uint8_t* meta;    // tiled metadata
  const float* sx;
  const float* sw;
  const uint16_t* bias;  // bf16 [N] added to every output row, or null
  int M, N, K;
  // batch (one-CTA kernel): L problems of the same shape; per-problem
  // offsets of the weight storage (bytes), scales (floats) and bias (values)
  int L;
  int64_t bs_values, bs_meta, bs_sx, bs_sw, bs_bias;
  int ldsx, ldsw;          // row strides (floats) of the scale tensors
  int gM_shift, gN_shift;  // log2 of the granularities (0 or 7)
  int m_tiles, n_tiles, k_tiles;
  int side_ksteps;  // r / 16
  // stream-K (one-CTA kernel, SPLIT instances): the stage sequence of all
  // tiles, tile-major, cut into one contiguous range per CTA
  int kst;          // stages per tile
  int cs;           // cluster split: CTAs of a cluster sharing one tile's K range (1 = none)
  int64_t sk_units; // stages in all (tiles x kst)
  float* ws;        // per CTA: one unscaled fp32 partial [BN][128]
  unsigned long long* flags;  // per CTA: the epoch at which its partial was published
  unsigned long long* sk_word;  // launch counter: epoch << 20 | CTAs that finished this launch
  unsigned int* err;
};

namespace {

constexpr int BM = 128;                  // weight rows per tile (MMA M)
constexpr int BK = 128;                  // logical K per stage (two sparse MMAs of K = 64)
constexpr int A_STAGE = BM * BK / 2;     // kept values: one 8 KB storage tile
constexpr int META_STAGE = BM * BK / 8;  // metadata: one 2 KB storage tile
constexpr int META_COL0 = 448;           // TMEM columns 448..511: metadata ring
constexpr int META_SLOTS = 16;           // 4 columns each
constexpr int MAX_STAGES = 16;
constexpr int PRODUCERS = 2;             // load warps; warp p issues the stages p, p + 2, ...
constexpr int MMA_WARP = PRODUCERS;
constexpr int EPI_WARP0 = PRODUCERS + 1;
constexpr int EPI_WARPS = 8;             // two per TMEM lane quadrant, each half of the columns
constexpr int EPI_THREADS = 32 * EPI_WARPS;
constexpr int NUM_THREADS = 32 * EPI_WARP0 + EPI_THREADS;
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int BAR_BYTES = 1024;

// Barrier over the epilogue threads (named barrier 1) that also ORs a
// predicate across them, so that a give-up decision is taken by all or none.
__device__ __forceinline__ bool epilogue_bar_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(EPI_THREADS)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory"); }

// Writes the four bf16 in (lo, hi) to dst[0], dst[stride], dst[2 stride], dst[3 stride].
__device__ __forceinline__ void st_bf16x4(uint16_t* dst, int stride, uint32_t lo, uint32_t hi) {
  dst[0] = static_cast<uint16_t>(lo & 0xFFFFu);
  dst[stride] = static_cast<uint16_t>(lo >> 16);
  dst[2 * stride] = static_cast<uint16_t>(hi & 0xFFFFu);
  dst[3 * stride] = static_cast<uint16_t>(hi >> 16);
}
// The bias of output channel n as fp32, or -0.0 without a bias: adding -0.0
// (or folding it into an FMA) leaves every value, the sign of zero included,
// exactly as it was.
__device__ __forceinline__ float bias_of(const GemmArgs& p, int n) {
  return p.bias ? __uint_as_float(static_cast<uint32_t>(__ldg(&p.bias[n])) << 16) : -0.0f;
}
// bf16((s_t sw) acc_t + add_t + bias) for 4 consecutive tokens t; s points at
// their 4 scales (16-byte aligned shared memory, the same address in every lane).
template <bool ADD>
__device__ __forceinline__ void scale4_store(const float* s, float sw, const uint32_t* acc, const uint32_t* add,
                                             float bias, uint16_t* dst, int stride) {
  const float4 s4 = *reinterpret_cast<const float4*>(s);
  const float2 b2 = make_float2(bias, bias);
  const float2 a01 = ADD ? __fadd2_rn(make_float2(__uint_as_float(add[0]), __uint_as_float(add[1])), b2) : b2;
  const float2 a23 = ADD ? __fadd2_rn(make_float2(__uint_as_float(add[2]), __uint_as_float(add[3])), b2) : b2;
  // packed pairs (sx sw, then times acc plus the addend): each value rounded as the scalar forms would
  const float2 w2 = make_float2(sw, sw);
  const float2 y01 = __ffma2_rn(__fmul2_rn(make_float2(s4.x, s4.y), w2),
                                make_float2(__uint_as_float(acc[0]), __uint_as_float(acc[1])), a01);
  const float2 y23 = __ffma2_rn(__fmul2_rn(make_float2(s4.z, s4.w), w2),
                                make_float2(__uint_as_float(acc[2]), __uint_as_float(acc[3])), a23);
  st_bf16x4(dst, stride, bf16x2_rn(y01.x, y01.y), bf16x2_rn(y23.x, y23.y));
}

// Loads `N8 * 8` consecutive accumulator columns of this warp's lanes.
template <int N8>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (N8 % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N8 / 2; ++i) tmem_ld16(taddr + 16 * i, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * i));
  } else {
#pragma unroll
    for (int i = 0; i < N8; ++i) tmem_ld8(taddr + 8 * i, r + 8 * i);
  }
}

}  // namespace

// Global-memory publish/observe of a 64-bit flag (release/acquire at GPU scope).
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// SM-pair kernel (sp24_gemm_pair.cu): per-token x per-channel scaling (gK =
// K), 256 weight rows x 256 tokens per pair tile, or x 240 tokens with the
// fused side GEMM (r <= 64).  pair_gemm_applies says whether a call takes it;
// launch_pair_gemm builds its tensor maps and launches it (args: operands,
// scales, sizes and the error word; tile counts are its own).
bool pair_gemm_applies(int64_t M, int64_t N, int64_t K, bool plain, int64_t r);
// Token tile of a plain-scaled pair launch (256 or 240) on a part with sm_count SMs.
int pair_token_tile(int64_t M, int64_t N, int sm_count);
sp24_status launch_pair_gemm(const DeviceInfo* dev, const void* Xq, int64_t ldx, const void* Y, int64_t ldy,
                             const void* X2, const void* W2, int64_t r, const GemmArgs& args, cudaStream_t stream);
// The same kernel with group-wise promotion (gK = 128): 256 weight rows x 128
// (or 112) tokens per pair tile, each K block's partial sum in one of three
// (or four) TMEM accumulators and scaled into fp32 registers by its epilogue.
bool pair_promote_applies(int64_t M, int64_t N, int64_t K, int64_t r);
// Token tile of a group-wise pair launch (128, or 112 with four accumulators).
int pair_promote_token_tile(int64_t M, int64_t N, int sm_count);
sp24_status launch_pair_promote(const DeviceInfo* dev, const void* Xq, int64_t ldx, const void* Y, int64_t ldy,
                                const GemmArgs& args, cudaStream_t stream);

}  // namespace sp24
