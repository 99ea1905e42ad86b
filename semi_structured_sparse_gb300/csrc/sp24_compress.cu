// sp24_compress.cu -- weight compression (magnitude 2:4 prune + e4m3 +
// pack) and dynamic activation quantization.  Both are HBM-bound streaming
// kernels: 16-byte vector loads, warp-level reductions, register-held rows,
// one pass over the input.
//
// Weight path: pytorch/ao PR #3258 ("Introduce new W8A8-FP-CSR quantization
// API", jcaip's review): drop the two smallest |w| of every group of four
// along K, positive amax-based scale, store only the kept values and the
// 2-bit metadata; all-zero weights are legal.  Scale granularities 1 x K,
// 1 x 128 and 128 x 128 follow CUTLASS PR #2095 ("Improvements for:
// Groupwise scaling along M for FP8 gemm", ScaleGranularity description).
// Activation path: same PR #3258, the activation is divided by its scale and
// cast to e4m3.
#include <cuda_bf16.h>
#include "sp24_internal.cuh"
#include "sp24_ptx.cuh"

namespace sp24 {
namespace {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// int8 sibling: symmetric codes in [-127, 127] (pytorch/ao PR #3258 names
// the int8 x int8 2:4 kernels; the quantizer is the plain symmetric one).
constexpr float kInt8Max = 127.0f;

// Scale for a block whose largest |w| has bf16 magnitude bits `amax_bits`:
// amax / 448 (amax / 127 for int8 codes), correctly rounded, or 1 when the
// block is all zeros.
template <bool I8 = false>
__device__ __forceinline__ float weight_scale(uint32_t amax_bits) {
  return amax_bits == 0 ? 1.0f : __fdiv_rn(bf16_bits_to_float(amax_bits), I8 ? kInt8Max : kE4M3Max);
}

// Running max of |w| over 16-byte chunks, kept as a packed bf16 pair: for
// finite bf16 the order of |w| is the order of the magnitude bits, so the
// packed bf16 max (on the half-precision pipe, beside the integer work of the
// packing) gives the same result as an integer max of the magnitude bits.
__device__ __forceinline__ uint32_t amax2_acc(uint32_t acc, const uint4& v) {
  const __nv_bfloat162 a = __hmax2(__habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.x)),
                                   __habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.y)));
  const __nv_bfloat162 b = __hmax2(__habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.z)),
                                   __habs2(*reinterpret_cast<const __nv_bfloat162*>(&v.w)));
  const __nv_bfloat162 m = __hmax2(__hmax2(a, b), *reinterpret_cast<const __nv_bfloat162*>(&acc));
  return *reinterpret_cast<const uint32_t*>(&m);
}
// Magnitude bits of the larger half of a packed pair from amax2_acc.
__device__ __forceinline__ uint32_t amax2_bits(uint32_t acc) { return max(acc & 0x7FFFu, (acc >> 16) & 0x7FFFu); }

// Largest bf16 magnitude (sign cleared) among the 8 values of a 16-byte
// chunk, with packed 16-bit unsigned max.
__device__ __forceinline__ uint32_t chunk_amax_bits(const uint4& v) {
  const uint32_t m2 = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m2 & 0xFFFFu, m2 >> 16);
}

// x / s, correctly rounded, given r = RN(1/s): Markstein's correction step
// (P. W. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(x r) is
// within an ulp of the quotient, the residual x - s q0 is exact in one FMA,
// and RN(q0 + residual r) is the correctly rounded x / s.  One reciprocal
// per row replaces a full division per element.  Conditions: every quotient
// here is at most 448 in magnitude (|x| <= amax = 448 s), so nothing
// overflows; the scale must be at least kMinFastScale, so that r is finite
// and, for any quotient that can round to a nonzero e4m3 code (>= 2^-10), the
// residual stays in the fp32 normal range (rows below it divide exactly).
// The sign is copied from x: for x = -0 the residual sum gives +0.
constexpr float kMinFastScale = 8.0779356e-28f;  // 2^-90
// The residual is formed as q0 s - x (the negated residual, equally exact)
// and the correction as q0 - that * r: for x = -0 this keeps q = -0 (with the
// residual taken as x - q0 s the sum +0 + -0 would give +0), so no separate
// sign fix is needed; for every other x the two forms compute the same
// correctly rounded quotient.
__device__ __forceinline__ float div_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float nrem = __fmaf_rn(q0, s, -x);
  return __fmaf_rn(-nrem, r, q0);
}

// Two fp32 -> int8 codes: nearest integer, ties to even, clamped to
// [-127, 127]; `lo` in bits [7:0], `hi` in bits [15:8].
__device__ __forceinline__ uint32_t to_s8x2(float lo, float hi) {
  const int a = max(-127, min(127, __float2int_rn(lo)));
  const int b = max(-127, min(127, __float2int_rn(hi)));
  return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8);
}

// Two fp32 -> e4m3 conversions in one instruction (round to nearest even,
// saturate to +-448); `lo` lands in bits [7:0], `hi` in bits [15:8].
__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Select, quantize and pack one group of four bf16 values held as two
// packed words: lo = (w1 << 16) | w0 and hi = (w3 << 16) | w2.
// Each element gets the key  |w| << 2 | (3 - i):  a larger key is a larger
// magnitude, and among equal magnitudes the lower index.  The two largest
// keys (a 4-input max/min network) are the two kept elements.  Their bf16
// bits are then pulled out of the 8 input bytes with one byte permute.
// Returns the two e4m3 codes in ascending position in bits [15:0] and the
// metadata nibble i0 | i1 << 2 in bits [19:16].
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
template <bool FAST, int NIB_SHIFT = 16, bool I8 = false>
__device__ __forceinline__ uint32_t pack_group(uint32_t lo, uint32_t hi, float s, float r) {
  // Keys from the raw words, with multiplies only (the FMA pipe, beside the
  // integer min/max work): a multiply by 2^17 moves an element's 15
  // magnitude bits to [31:17] and pushes its sign bit and the neighbouring
  // element out of the word, so no |w| or mask step is needed; the added
  // 3 - i fills bits [1:0].  The high half is brought down first with a
  // high multiply (x >> 16).
  const uint32_t k0 = lo * (1u << 17) + 3u;                    // element 0
  const uint32_t k1 = __umulhi(lo, 1u << 16) * (1u << 17) + 2u;  // element 1
  const uint32_t k2 = hi * (1u << 17) + 1u;                    // element 2
  const uint32_t k3 = __umulhi(hi, 1u << 16) * (1u << 17);       // element 3
  const uint32_t hi01 = max(k0, k1), lo01 = min(k0, k1);
  const uint32_t hi23 = max(k2, k3), lo23 = min(k2, k3);
  const uint32_t first = max(hi01, hi23);
  const uint32_t second = max(min(hi01, hi23), max(lo01, lo23));
  const uint32_t ia = (first & 3u) ^ 3u, ib = (second & 3u) ^ 3u;
  const uint32_t i0 = min(ia, ib), i1 = max(ia, ib);
  // byte selector: element i is bytes 2i, 2i+1 of {hi:lo}; kept pair -> {v_i1 : v_i0}
  const uint32_t sel = i0 * 0x22u + i1 * 0x2200u + 0x1010u;
  const uint32_t pair = prmt(lo, hi, sel);
  const float x0 = __uint_as_float(pair * 65536u), x1 = __uint_as_float(__umulhi(pair, 65536u) * 65536u);
  const float q0 = FAST ? div_scale(x0, s, r) : __fdiv_rn(x0, s);
  const float q1 = FAST ? div_scale(x1, s, r) : __fdiv_rn(x1, s);
  const uint32_t q = I8 ? to_s8x2(q0, q1) : to_e4m3x2(q0, q1);
  // q < 2^16: the nibble i0 | i1 << 2 goes to bits [NIB_SHIFT + 3 : NIB_SHIFT]
  return q + i0 * (1u << NIB_SHIFT) + i1 * (4u << NIB_SHIFT);
}

// Two groups (8 bf16 in a 16-byte chunk) -> 4 value bytes and 1 meta byte.
template <bool FAST, bool I8 = false>
__device__ __forceinline__ void pack_chunk(const uint4& v, float s, float r, uint32_t& vals, uint32_t& metab) {
  const uint32_t g0 = pack_group<FAST, 16, I8>(v.x, v.y, s, r);  // nibble in bits [19:16]
  const uint32_t g1 = pack_group<FAST, 20, I8>(v.z, v.w, s, r);  // nibble in bits [23:20]
  vals = prmt(g0, g1, 0x5410u);           // codes of group 0 in bytes 0-1, group 1 in bytes 2-3
  metab = prmt(g0 | g1, 0u, 0x4442u);     // byte 2 of (g0 | g1): the two nibbles
}

// Storage the GEMM reads (see sp24.h): 128-row x 128-K tiles, tile-contiguous,
// consecutive along K within a 128-row band; kept values with the 64-byte
// swizzle applied inside a tile.  Offsets of 4 kept bytes starting at kept
// index j (j % 4 == 0) of row n, and of meta byte jb of row n.
__device__ __forceinline__ int64_t values_offset(int n, int j, int K) {
  const int64_t t = static_cast<int64_t>(n >> 7) * (K >> 7) + (j >> 6);
  const int r = n & 127, b = j & 63;
  return t * 8192 + r * 64 + (((b >> 4) ^ ((r >> 1) & 3)) << 4) + (b & 15);
}
__device__ __forceinline__ int64_t meta_offset(int n, int jb, int K) {
  const int64_t t = static_cast<int64_t>(n >> 7) * (K >> 7) + (jb >> 4);
  return t * 2048 + (n & 127) * 16 + (jb & 15);
}

// Per-lane parts of those offsets for the row kernels, where lane l of a warp
// packs the 8 weights at k = 256 c + 8 l: its 4 value bytes land in tile
// 2c + l/16 and its meta byte in the same tile; chunk c adds 2 tiles.
struct RowStore {
  int64_t v, m;  // offsets for chunk 0
  __device__ RowStore(int n, int K, int lane) {
    const int r = n & 127;
    const int64_t band = static_cast<int64_t>(n >> 7) * (K >> 7);
    v = band * 8192 + (lane >> 4) * 8192 + r * 64 + ((((lane & 15) >> 2) ^ ((r >> 1) & 3)) << 4) + (lane & 3) * 4;
    m = band * 2048 + (lane >> 4) * 2048 + r * 16 + (lane & 15);
  }
  __device__ int64_t values_at(int c) const { return v + static_cast<int64_t>(c) * 16384; }
  __device__ int64_t meta_at(int c) const { return m + static_cast<int64_t>(c) * 4096; }
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Packs and stores the chunks c = h, h + WPR, ... of row n (WPR warps per
// row): the first kHeldChunks from registers, any further ones re-read from
// global.
template <bool FAST, int WPR, bool I8 = false>
__device__ __forceinline__ void emit_row(const uint4 (&held)[8], const uint16_t* row, int n, int K, int nchunks, int h,
                                         int lane, float s, float r, uint8_t* values, uint8_t* meta) {
  const RowStore st(n, K, lane);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = WPR * i + h, k = c * 256 + lane * 8;
    if (c < nchunks && k < K) {
      uint32_t vals, mb;
      pack_chunk<FAST, I8>(held[i], s, r, vals, mb);
      *reinterpret_cast<uint32_t*>(values + st.values_at(c)) = vals;
      meta[st.meta_at(c)] = static_cast<uint8_t>(mb);
    }
  }
  for (int c = 8 * WPR + h; c < nchunks; c += WPR) {
    const int k = c * 256 + lane * 8;
    if (k < K) {
      uint32_t vals, mb;
      pack_chunk<FAST, I8>(*reinterpret_cast<const uint4*>(row + k), s, r, vals, mb);
      *reinterpret_cast<uint32_t*>(values + st.values_at(c)) = vals;
      meta[st.meta_at(c)] = static_cast<uint8_t>(mb);
    }
  }
}

constexpr int kRowsPerCta = 8;   // gK = 128: one warp per weight row
constexpr int kRowThreads = 128;    // gK = K: 128-thread CTAs (a finer last wave), WPR warps per weight row
constexpr int kHeldChunks = 8;   // per warp: 8 x 16 bytes per lane stay in registers

// gN = 1.  GK128 = false: one scale per row (gK = K), rows longer than 4096
// (shorter ones take compress_rows_pipe_kernel); WPR warps share a row (4 up
// to K = 8192, 8 above, so that every chunk of rows up to 16384 stays in
// registers), warp h owning the 256-element chunks c = h, h + WPR, ...; the
// row's amax is combined through shared memory.
// GK128 = true: one scale per row and 128-wide K block; one warp per row,
// each half-warp owns a block.
template <bool GK128, int WPR = 2, bool I8 = false>
__global__ void __launch_bounds__(256, 4) compress_rows_kernel(const uint16_t* __restrict__ W, int N, int K, int64_t ldw,
                                                            uint8_t* __restrict__ values, uint8_t* __restrict__ meta,
                                                            float* __restrict__ scales) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = (K + 255) / 256;  // 256 elements per warp step, 8 per lane
  pdl_wait();

  if (!GK128) {
    __shared__ uint32_t warp_amax[8];
    const int h = warp % WPR;
    const int n = blockIdx.x * (blockDim.x / 32 / WPR) + warp / WPR;
    const bool valid = n < N;
    const uint16_t* row = W + static_cast<int64_t>(valid ? n : 0) * ldw;
    uint4 held[kHeldChunks];
    uint32_t amax2 = 0;
#pragma unroll
    for (int i = 0; i < kHeldChunks; ++i) {
      const int c = WPR * i + h, k = c * 256 + lane * 8;
      if (valid && c < nchunks && k < K) {
        held[i] = ldg_stream(row + k);
        amax2 = amax2_acc(amax2, held[i]);
      }
    }
    for (int c = WPR * kHeldChunks + h; valid && c < nchunks; c += WPR) {  // longer rows: stream for amax
      const int k = c * 256 + lane * 8;
      if (k < K) amax2 = amax2_acc(amax2, ldg_stream(row + k));
    }
    uint32_t amax = __reduce_max_sync(0xFFFFFFFFu, amax2_bits(amax2));
    if (lane == 0) warp_amax[warp] = amax;
    __syncthreads();
    if (!valid) return;
    const int w0 = warp - h;  // the row's first warp
#pragma unroll
    for (int i = 0; i < WPR; ++i) amax = max(amax, warp_amax[w0 + i]);
    const float s = weight_scale<I8>(amax), r = __frcp_rn(s);
    if (lane == 0 && h == 0) scales[n] = s;
    if (s >= kMinFastScale)  // the same for the whole row: warp-uniform
      emit_row<true, WPR, I8>(held, row, n, K, nchunks, h, lane, s, r, values, meta);
    else
      emit_row<false, WPR, I8>(held, row, n, K, nchunks, h, lane, s, r, values, meta);
  } else {
    // lanes 0-15 cover K block 2c, lanes 16-31 block 2c+1 (when it exists)
    const int n = blockIdx.x * kRowsPerCta + warp;
    if (n >= N) return;
    const uint16_t* row = W + static_cast<int64_t>(n) * ldw;
    const RowStore st(n, K, lane);
    for (int c = 0; c < nchunks; ++c) {
      const int k = c * 256 + lane * 8;
      const bool active = k < K;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (active) v = ldg_stream(row + k);
      uint32_t amax = active ? chunk_amax_bits(v) : 0u;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      const float s = weight_scale(amax), r = __frcp_rn(s);
      if (active) {
        if ((lane & 15) == 0) scales[static_cast<int64_t>(k / 128) * N + n] = s;
        uint32_t vals, mb;
        if (s >= kMinFastScale)
          pack_chunk<true>(v, s, r, vals, mb);
        else
          pack_chunk<false>(v, s, r, vals, mb);
        *reinterpret_cast<uint32_t*>(values + st.values_at(c)) = vals;
        meta[st.meta_at(c)] = static_cast<uint8_t>(mb);
      }
    }
  }
  pdl_trigger();
}

// gN = 1, gK = K, K <= 4096: persistent warp pairs.  Pair p of the grid walks
// rows p, p + P, p + 2P, ... (P pairs in all; pair p is pair p / G of CTA
// p mod G, G CTAs); warp h of a pair owns the
// chunks c = h, h + 2, ... of a row, all held in registers, and loads its
// chunks of the pair's next row before it packs the current one, so that
// the loads of one row overlap the integer work of the previous (with every
// row's loads issued at once, a row could only be packed once its last
// chunk had arrived).  The pair combines its row amax through shared memory
// (one slot per row parity) and a named barrier of its 64 threads.
template <int PAIRS, bool I8 = false>
__global__ void __launch_bounds__(64 * PAIRS, 1) compress_rows_pipe_kernel(const uint16_t* __restrict__ W, int N, int K,
                                                                         int64_t ldw, uint8_t* __restrict__ values,
                                                                         uint8_t* __restrict__ meta,
                                                                         float* __restrict__ scales) {
  __shared__ uint32_t pair_amax[PAIRS][2][2];  // [pair][row parity][warp of the pair]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pr = warp >> 1, h = warp & 1;
  const int stride = gridDim.x * PAIRS;
  const int nchunks = (K + 255) / 256;  // at most 16: 8 per warp
  pdl_wait();
  auto load = [&](int n, uint4 (&held)[8]) {
    const uint16_t* row = W + static_cast<int64_t>(n) * ldw;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 2 * i + h, k = c * 256 + lane * 8;
      if (c < nchunks && k < K) held[i] = ldg_stream(row + k);
    }
  };
  // one row: amax, scale, packing; it is the pair's parity-th row
  auto pack = [&](int n, int parity, const uint4 (&held)[8]) {
    uint32_t amax2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 2 * i + h, k = c * 256 + lane * 8;
      if (c < nchunks && k < K) amax2 = amax2_acc(amax2, held[i]);
    }
    const uint32_t amax_w = __reduce_max_sync(0xFFFFFFFFu, amax2_bits(amax2));
    if (lane == 0) pair_amax[pr][parity][h] = amax_w;
    asm volatile("bar.sync %0, 64;" ::"r"(1 + pr) : "memory");
    const uint32_t amax = max(pair_amax[pr][parity][0], pair_amax[pr][parity][1]);
    const float s = weight_scale<I8>(amax), r = __frcp_rn(s);
    if (lane == 0 && h == 0) scales[n] = s;
    const uint16_t* row = W + static_cast<int64_t>(n) * ldw;
    if (s >= kMinFastScale)  // the same for the whole row: pair-uniform
      emit_row<true, 2, I8>(held, row, n, K, nchunks, h, lane, s, r, values, meta);
    else
      emit_row<false, 2, I8>(held, row, n, K, nchunks, h, lane, s, r, values, meta);
  };
  uint4 a[8], b[8];
  // pair pr of CTA c is pair pr G + c of the grid: when the rows do not divide
  // evenly, the pairs with one row more are spread over all the SMs instead
  // of filling the first CTAs (4096 rows: 448 of 1216 pairs take a fourth)
  int n = pr * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  if (n < N) load(n, a);
  // two rows per trip, so that the two row buffers keep their registers
  for (; n < N; n += 2 * stride) {
    if (n + stride < N) load(n + stride, b);
    pack(n, 0, a);
    if (n + stride >= N) break;
    if (n + 2 * stride < N) load(n + 2 * stride, a);
    pack(n + stride, 1, b);
  }
  pdl_trigger();
}

// gN = gK = 128: one CTA of 256 threads per 128 x 128 block.  Thread t owns
// columns 8*(t%16) .. +7 of rows t/16 + 16*i, i = 0..7.
__global__ void __launch_bounds__(256) compress_blocks_kernel(const uint16_t* __restrict__ W, int N, int K,
                                                              int64_t ldw, uint8_t* __restrict__ values,
                                                              uint8_t* __restrict__ meta,
                                                              float* __restrict__ scales) {
  __shared__ uint32_t warp_max[8];
  const int kb = blockIdx.x, nb = blockIdx.y;
  const int t = threadIdx.x, cseg = t & 15, r0 = t >> 4;
  const int k = kb * 128 + cseg * 8;
  pdl_wait();
  uint4 v[8];
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = nb * 128 + r0 + 16 * i;
    v[i] = ldg_stream(W + static_cast<int64_t>(n) * ldw + k);
    amax = max(amax, chunk_amax_bits(v[i]));
  }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
  if ((t & 31) == 0) warp_max[t >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = max(amax, warp_max[w]);
  const float s = weight_scale(amax), r = __frcp_rn(s);
  if (t == 0) scales[static_cast<int64_t>(kb) * (N / 128) + nb] = s;
  // The block is exactly one storage tile, and rows r0 + 16 i share the
  // swizzle of row r0 (it depends on (row / 2) mod 4): the stores of row
  // r0 + 16 i land 16 * 64 bytes (values) and 16 * 16 bytes (metadata) after
  // those of row r0.
  uint8_t* vrow = values + values_offset(nb * 128 + r0, k / 2, K);
  uint8_t* mrow = meta + meta_offset(nb * 128 + r0, k / 8, K);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t vals, mb;
    if (s >= kMinFastScale)  // the same for the whole block: CTA-uniform
      pack_chunk<true>(v[i], s, r, vals, mb);
    else
      pack_chunk<false>(v[i], s, r, vals, mb);
    *reinterpret_cast<uint32_t*>(vrow + i * 1024) = vals;
    mrow[i * 256] = static_cast<uint8_t>(mb);
  }
  pdl_trigger();
}

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Activation quantization (fp32 input): one warp per token row; 128
// elements per warp step (4 per lane).  GK128: each step is one scale block.
template <bool GK128, bool I8 = false>
__global__ void __launch_bounds__(256) quantize_act_kernel(const float* __restrict__ X, int M, int K, int64_t ldx,
                                                           uint8_t* __restrict__ xq, float* __restrict__ sx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * 8 + warp;
  pdl_wait();
  if (m >= M) return;
  const float* row = X + static_cast<int64_t>(m) * ldx;
  uint8_t* qrow = xq + static_cast<int64_t>(m) * K;
  const int nsteps = K / 128;
  auto quant4 = [&](const float4& f, float s) -> uint32_t {
    if (I8)
      return to_s8x2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s)) | (to_s8x2(__fdiv_rn(f.z, s), __fdiv_rn(f.w, s)) << 16);
    return to_e4m3x2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s)) | (to_e4m3x2(__fdiv_rn(f.z, s), __fdiv_rn(f.w, s)) << 16);
  };
  constexpr float kQMax = I8 ? kInt8Max : kE4M3Max;
  auto amax4 = [](const float4& f) { return fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))); };
  if (GK128) {
    for (int c = 0; c < nsteps; ++c) {
      const float4 f = load4(row + c * 128 + lane * 4);
      float a = amax4(f);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
      const float s = a == 0.0f ? 1.0f : __fdiv_rn(a, kQMax);
      if (lane == 0) sx[static_cast<int64_t>(c) * M + m] = s;
      *reinterpret_cast<uint32_t*>(qrow + c * 128 + lane * 4) = quant4(f, s);
    }
  } else {
    float a = 0.0f;
    for (int c = 0; c < nsteps; ++c) a = fmaxf(a, amax4(load4(row + c * 128 + lane * 4)));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
    const float s = a == 0.0f ? 1.0f : __fdiv_rn(a, kQMax);
    if (lane == 0) sx[m] = s;
    for (int c = 0; c < nsteps; ++c) {
      const float4 f = load4(row + c * 128 + lane * 4);
      *reinterpret_cast<uint32_t*>(qrow + c * 128 + lane * 4) = quant4(f, s);
    }
  }
  pdl_trigger();
}

}  // namespace
}  // namespace sp24

extern "C" sp24_status sp24_fp8_compress(const void* W, int64_t N, int64_t K, int64_t ldw, int gN, int gK,
                                         void* values, void* meta, float* scales, void* stream) {
  using namespace sp24;
  if (!W || !values || !meta || !scales) return SP24_ERR_INVALID_ARG;
  if (N < 1 || K < 128 || K % 128 != 0 || ldw < K || N > (1 << 30) || K > (1 << 30)) return SP24_ERR_INVALID_ARG;
  const bool per_channel = (gN == 1 && gK == K);
  const bool row_k128 = (gN == 1 && gK == 128);
  const bool block128 = (gN == 128 && gK == 128);
  if (!per_channel && !row_k128 && !block128) return SP24_ERR_UNSUPPORTED;
  if (N % 128 != 0) return SP24_ERR_INVALID_ARG;  // tiled storage: whole 128-row bands
  if (!aligned16(W) || !aligned16(values) || !aligned16(meta) || (ldw * 2) % 16 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(scales) % 4 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* w = static_cast<const uint16_t*>(W);
  uint8_t* v = static_cast<uint8_t*>(values);
  uint8_t* m = static_cast<uint8_t*>(meta);
  if (block128) {
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
    if (grid.y > 65535u) return SP24_ERR_UNSUPPORTED;
    if (launch_pdl(compress_blocks_kernel, grid, dim3(256), 0, s, w, (int)N, (int)K, ldw, v, m, scales) !=
        cudaSuccess)
      return SP24_ERR_CUDA;
  } else {
    if (per_channel && K <= 4096) {
      // persistent warp pairs, one CTA of 8 pairs per SM (fewer when N is small)
      constexpr int kPairs = 8;
      const int64_t ctas = (N + kPairs - 1) / kPairs;
      const unsigned grid = static_cast<unsigned>(ctas < dev->sm_count ? ctas : dev->sm_count);
      if (launch_pdl(compress_rows_pipe_kernel<kPairs>, dim3(grid), dim3(64 * kPairs), 0, s, w, (int)N, (int)K, ldw, v,
                     m, scales) != cudaSuccess)
        return SP24_ERR_CUDA;
    } else if (per_channel) {
      // warps per row: enough to hold a row of up to 16384 in registers
      const int wpr = K <= 8192 ? 4 : 8;
      const int rows_per_cta = wpr <= 4 ? kRowThreads / 32 / wpr : 1;
      const unsigned threads = wpr <= 4 ? kRowThreads : 256;
      const unsigned grid = static_cast<unsigned>((N + rows_per_cta - 1) / rows_per_cta);
      cudaError_t e;
      if (wpr == 4)
        e = launch_pdl(compress_rows_kernel<false, 4>, dim3(grid), dim3(threads), 0, s, w, (int)N, (int)K, ldw, v, m,
                       scales);
      else
        e = launch_pdl(compress_rows_kernel<false, 8>, dim3(grid), dim3(threads), 0, s, w, (int)N, (int)K, ldw, v, m,
                       scales);
      if (e != cudaSuccess) return SP24_ERR_CUDA;
    } else {
      const unsigned grid = static_cast<unsigned>((N + kRowsPerCta - 1) / kRowsPerCta);
      if (launch_pdl(compress_rows_kernel<true>, dim3(grid), dim3(256), 0, s, w, (int)N, (int)K, ldw, v, m,
                     scales) != cudaSuccess)
        return SP24_ERR_CUDA;
    }
  }
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

namespace sp24 {
namespace {

// Two e4m3 codes (low byte first) as floats: e4m3 -> f16 is exact, f16 -> f32 too.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t codes) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(codes)));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The dense dequantized weight from the library's storage: W[n][k] =
// bf16(sw * decode(value)) at the two kept positions of every group of four,
// 0 at the other two -- what the GEMM returns for an identity activation
// (pytorch/ao PR #3258, dequantize by multiplying with an identity), without
// the GEMM.  One warp per row and 1024 consecutive k: each lane expands one
// 16-byte chunk of kept values and 4 metadata bytes into 64 output bytes.
__global__ void __launch_bounds__(256) decompress_kernel(const uint8_t* __restrict__ values,
                                                         const uint8_t* __restrict__ meta,
                                                         const float* __restrict__ scales, int N, int K, int gN_shift,
                                                         int gK, int ldsc, uint16_t* __restrict__ W, int64_t ldw) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  const int k0 = blockIdx.y * 1024 + lane * 32;
  pdl_wait();
  if (n >= N || k0 >= K) return;
  const uint4 v = *reinterpret_cast<const uint4*>(values + values_offset(n, k0 / 2, K));
  const uint32_t mw = *reinterpret_cast<const uint32_t*>(meta + meta_offset(n, k0 / 8, K));
  const float s = scales[static_cast<int64_t>(k0 / gK) * ldsc + (n >> gN_shift)];
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[16];  // 32 bf16, two per word
#pragma unroll
  for (int g = 0; g < 8; ++g) {  // weights k0 + 4g + [0, 4): kept values 2g (position i0) and 2g + 1 (i1 > i0)
    const uint32_t nib = (mw >> (4 * g)) & 0xFu;
    const uint32_t i0 = nib & 3u, i1 = nib >> 2;
    const float2 f = e4m3x2_to_float2(vw[g / 2] >> (16 * (g & 1)));
    const uint32_t b = bf16x2_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
    const uint32_t b0 = b & 0xFFFFu, b1 = b >> 16;
    out[2 * g] = (i0 < 2 ? b0 << (16 * i0) : 0u) | (i1 < 2 ? b1 << (16 * i1) : 0u);
    out[2 * g + 1] = (i0 >= 2 ? b0 << (16 * (i0 - 2)) : 0u) | (i1 >= 2 ? b1 << (16 * (i1 - 2)) : 0u);
  }
  uint4* dst = reinterpret_cast<uint4*>(W + static_cast<int64_t>(n) * ldw + k0);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
  pdl_trigger();
}

// x / s for 8 bf16 values (one 16-byte chunk) as 8 e4m3 codes, with the
// correctly rounded division of the weight path (div_scale; exact division
// for scales below kMinFastScale, where the reciprocal would overflow).
__device__ __forceinline__ uint2 quant8(const uint4& v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t q[4];
  if (s >= kMinFastScale) {
    const float r = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      q[i] = to_e4m3x2(div_scale(bf16_bits_to_float(w[i] & 0xFFFFu), s, r), div_scale(bf16_bits_to_float(w[i] >> 16), s, r));
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      q[i] = to_e4m3x2(__fdiv_rn(bf16_bits_to_float(w[i] & 0xFFFFu), s), __fdiv_rn(bf16_bits_to_float(w[i] >> 16), s));
  }
  return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// Activation quantization from bf16 (the dtype of the pages' models): one
// CTA of 4 warps per token row; warp w takes the steps w, w + 4, ... of 256
// elements (one 16-byte load per lane), so a 128-wide scale block is a half
// warp.  Rows of up to 4096 elements stay in registers between the amax and
// the quantization; per token, the 4 warps' maxima meet in shared memory.
constexpr int kActWarps = 4;
constexpr int kHeldSteps = 4;  // per warp: K <= kActWarps * kHeldSteps * 256 = 4096 held
template <bool GK128>
__global__ void __launch_bounds__(32 * kActWarps) quantize_act_bf16_kernel(const uint16_t* __restrict__ X, int M,
                                                                           int K, int64_t ldx,
                                                                           uint8_t* __restrict__ xq,
                                                                           float* __restrict__ sx) {
  __shared__ uint32_t wmax[kActWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x;
  pdl_wait();
  const uint16_t* row = X + static_cast<int64_t>(m) * ldx;
  uint8_t* qrow = xq + static_cast<int64_t>(m) * K;
  const int nsteps = (K + 255) / 256;  // a last step of 128 elements uses lanes 0-15
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 held[kHeldSteps];
  uint32_t acc = 0;
#pragma unroll
  for (int i = 0; i < kHeldSteps; ++i) {
    const int c = warp + kActWarps * i, k = c * 256 + lane * 8;
    held[i] = (c < nsteps && k < K) ? ldg_stream(row + k) : zero;
    if (!GK128) acc = amax2_acc(acc, held[i]);
  }
  if (GK128) {
    auto block = [&](int c, const uint4& v) {  // one step: two 128-wide scale blocks, a half warp each
      const int k = c * 256 + lane * 8;
      uint32_t a = amax2_bits(amax2_acc(0u, v));
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
      const float s = weight_scale(a);
      if (k < K && (lane & 15) == 0) sx[static_cast<int64_t>(k / 128) * M + m] = s;
      if (k < K) *reinterpret_cast<uint2*>(qrow + k) = quant8(v, s);
    };
#pragma unroll
    for (int i = 0; i < kHeldSteps; ++i)
      if (warp + kActWarps * i < nsteps) block(warp + kActWarps * i, held[i]);
    for (int c = warp + kActWarps * kHeldSteps; c < nsteps; c += kActWarps) {
      const int k = c * 256 + lane * 8;
      block(c, k < K ? ldg_stream(row + k) : zero);
    }
  } else {
    for (int c = warp + kActWarps * kHeldSteps; c < nsteps; c += kActWarps) {
      const int k = c * 256 + lane * 8;
      if (k < K) acc = amax2_acc(acc, ldg_stream(row + k));
    }
    uint32_t a = amax2_bits(acc);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
    if (lane == 0) wmax[warp] = a;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kActWarps; ++w) a = max(a, wmax[w]);
    const float s = weight_scale(a);
    if (threadIdx.x == 0) sx[m] = s;
#pragma unroll
    for (int i = 0; i < kHeldSteps; ++i) {
      const int c = warp + kActWarps * i, k = c * 256 + lane * 8;
      if (c < nsteps && k < K) *reinterpret_cast<uint2*>(qrow + k) = quant8(held[i], s);
    }
    for (int c = warp + kActWarps * kHeldSteps; c < nsteps; c += kActWarps) {
      const int k = c * 256 + lane * 8;
      if (k < K) *reinterpret_cast<uint2*>(qrow + k) = quant8(ldg_stream(row + k), s);
    }
  }
  pdl_trigger();
}

template <typename T>
sp24_status quantize_act(const T* X, int64_t M, int64_t K, int64_t ldx, int gK, void* xq, float* sx, void* stream) {
  if (!X || !xq || !sx) return SP24_ERR_INVALID_ARG;
  if (M < 1 || K < 128 || K % 128 != 0 || ldx < K || M > (1 << 30) || K > (1 << 30)) return SP24_ERR_INVALID_ARG;
  if (gK != K && gK != 128) return SP24_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(xq) || (ldx * static_cast<int64_t>(sizeof(T))) % 16 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(sx) % 4 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>((M + 7) / 8);
  auto kern = [&](auto k, unsigned blocks, unsigned threads) {
    return launch_pdl(k, dim3(blocks), dim3(threads), 0, s, X, (int)M, (int)K, ldx, static_cast<uint8_t*>(xq),
                      sx) == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
  };
  if constexpr (sizeof(T) == 2) {
    const unsigned rows = static_cast<unsigned>(M), threads = 32 * kActWarps;
    st = gK == 128 ? kern(quantize_act_bf16_kernel<true>, rows, threads)
                   : kern(quantize_act_bf16_kernel<false>, rows, threads);
  } else {
    st = gK == 128 ? kern(quantize_act_kernel<true>, grid, 256) : kern(quantize_act_kernel<false>, grid, 256);
  }
  if (st != SP24_OK) return st;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

}  // namespace
}  // namespace sp24

extern "C" sp24_status sp24_fp8_quantize_act(const float* X, int64_t M, int64_t K, int64_t ldx, int gK, void* xq,
                                             float* sx, void* stream) {
  return sp24::quantize_act(X, M, K, ldx, gK, xq, sx, stream);
}

extern "C" sp24_status sp24_fp8_quantize_act_bf16(const void* X, int64_t M, int64_t K, int64_t ldx, int gK, void* xq,
                                                  float* sx, void* stream) {
  return sp24::quantize_act(static_cast<const uint16_t*>(X), M, K, ldx, gK, xq, sx, stream);
}

extern "C" sp24_status sp24_int8_compress(const void* W, int64_t N, int64_t K, int64_t ldw, void* values, void* meta,
                                          float* scales, void* stream) {
  using namespace sp24;
  if (!W || !values || !meta || !scales) return SP24_ERR_INVALID_ARG;
  if (N < 1 || K < 128 || K % 128 != 0 || ldw < K || N > (1 << 30) || K > (1 << 30)) return SP24_ERR_INVALID_ARG;
  if (N % 128 != 0) return SP24_ERR_INVALID_ARG;  // tiled storage: whole 128-row bands
  if (!aligned16(W) || !aligned16(values) || !aligned16(meta) || (ldw * 2) % 16 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(scales) % 4 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* w = static_cast<const uint16_t*>(W);
  uint8_t* v = static_cast<uint8_t*>(values);
  uint8_t* m = static_cast<uint8_t*>(meta);
  cudaError_t e;
  if (K <= 4096) {  // the FP8 path's kernels with int8 codes
    constexpr int kPairs = 8;
    const int64_t ctas = (N + kPairs - 1) / kPairs;
    const unsigned grid = static_cast<unsigned>(ctas < dev->sm_count ? ctas : dev->sm_count);
    e = launch_pdl(compress_rows_pipe_kernel<kPairs, true>, dim3(grid), dim3(64 * kPairs), 0, s, w, (int)N, (int)K,
                   ldw, v, m, scales);
  } else {
    const int wpr = K <= 8192 ? 4 : 8;
    const int rows_per_cta = wpr <= 4 ? kRowThreads / 32 / wpr : 1;
    const unsigned threads = wpr <= 4 ? kRowThreads : 256;
    const unsigned grid = static_cast<unsigned>((N + rows_per_cta - 1) / rows_per_cta);
    e = wpr == 4 ? launch_pdl(compress_rows_kernel<false, 4, true>, dim3(grid), dim3(threads), 0, s, w, (int)N, (int)K,
                              ldw, v, m, scales)
                 : launch_pdl(compress_rows_kernel<false, 8, true>, dim3(grid), dim3(threads), 0, s, w, (int)N, (int)K,
                              ldw, v, m, scales);
  }
  if (e != cudaSuccess) return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

extern "C" sp24_status sp24_int8_quantize_act(const float* X, int64_t M, int64_t K, int64_t ldx, void* xq, float* sx,
                                              void* stream) {
  using namespace sp24;
  if (!X || !xq || !sx) return SP24_ERR_INVALID_ARG;
  if (M < 1 || K < 128 || K % 128 != 0 || ldx < K || M > (1 << 30) || K > (1 << 30)) return SP24_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(xq) || (ldx * 4) % 16 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(sx) % 4 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  const sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_pdl(quantize_act_kernel<false, true>, dim3(static_cast<unsigned>((M + 7) / 8)), dim3(256), 0, s, X, (int)M,
                 (int)K, ldx, static_cast<uint8_t*>(xq), sx) != cudaSuccess)
    return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

extern "C" sp24_status sp24_fp8_decompress(const void* values, const void* meta, const float* scales, int64_t N,
                                           int64_t K, int gN, int gK, void* W, int64_t ldw, void* stream) {
  using namespace sp24;
  if (!values || !meta || !scales || !W) return SP24_ERR_INVALID_ARG;
  if (N < 1 || K < 128 || K % 128 != 0 || ldw < K || N > (1 << 30) || K > (1 << 30)) return SP24_ERR_INVALID_ARG;
  if (!((gN == 1 && gK == K) || (gN == 1 && gK == 128) || (gN == 128 && gK == 128))) return SP24_ERR_UNSUPPORTED;
  if (N % 128 != 0) return SP24_ERR_INVALID_ARG;  // tiled storage: whole 128-row bands
  if (!aligned16(values) || !aligned16(meta) || !aligned16(W) || (ldw * 2) % 16 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(scales) % 4 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;
  const dim3 grid(static_cast<unsigned>((N + 7) / 8), static_cast<unsigned>((K + 1023) / 1024));
  const int ldsc = static_cast<int>((N + gN - 1) / gN);
  if (launch_pdl(decompress_kernel, grid, dim3(256), 0, static_cast<cudaStream_t>(stream),
                 static_cast<const uint8_t*>(values), static_cast<const uint8_t*>(meta), scales, (int)N, (int)K,
                 gN == 128 ? 7 : 0, gK, ldsc, static_cast<uint16_t*>(W), ldw) != cudaSuccess)
    return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}
