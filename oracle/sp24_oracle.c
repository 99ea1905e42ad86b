/*
 * sp24_oracle.c -- plain CPU oracle for the 2:4 sparse FP8 linear-layer path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the package smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant generator with the CUDA implementation.
 *
 * What it computes, and where each step comes from:
 *   - magnitude 2:4 pruning along K: in every group of four consecutive K
 *     elements of a weight row, the two smallest magnitudes are zeroed
 *     (pytorch/ao PR #3258 "Introduce new W8A8-FP-CSR quantization API",
 *     jcaip's review of the pruning code: argsort of |w| over each group of
 *     four, the first two indices scattered to zero);
 *   - weight scale amax/448 per output channel or per 128x128 block, strictly
 *     positive (same PR, review thread on the positive-scale check; block
 *     granularity from CUTLASS PR #2095 "Improvements for: Groupwise scaling
 *     along M for FP8 gemm", ScaleGranularityM/N description);
 *   - e4m3 quantization q = e4m3(x / scale) (same PR, activation path that
 *     casts the scaled tensor to float8_e4m3fn), written here from the OCP
 *     FP8 E4M3 format definition (1 sign, 4 exponent bits with bias 7, 3
 *     mantissa bits, no infinities, S.1111.111 = NaN, max finite 448);
 *   - packing into kept values plus 2-bit position metadata, and nothing
 *     dense (same PR, jcaip: store specified values and sparsity metadata);
 *   - the group-wise scaled GEMM Y = X.W^T, each K block of length gK
 *     summed, then multiplied by sx*sw and added to the running sum (CUTLASS
 *     PR #2095, promotion of per-K-tile partial sums), plus an optional
 *     bf16 side GEMM X2.W2^T added into the same output (CUTLASS issue
 *     #2058 "How to implement a fused mixed precision matrix multiplication
 *     such as w4a4 + w16a16?", hyx1999's statement of Y = X1 W1^T + X2 W2^T);
 *   - the int8 x int8 2:4 sibling (same PR #3258, review: int8 x int8 and
 *     fp8 x fp8 are the two 2:4 kernels): symmetric int8 quantization of the
 *     pruned weight and the activation, exact integer sums (section at the
 *     end of this file).
 *
 * Readings taken where the pages are silent:
 *   - ties in the pruning argsort: the lower index wins;
 *   - amax == 0 (all-zero group, which must be accepted): scale = 1;
 *   - quantization divides by the scale (IEEE fp32, correctly rounded),
 *     then rounds to nearest-even with saturation to +-448; the sign of a
 *     value that rounds to zero is kept (0x80);
 *   - metadata nibble of a group = i0 | i1 << 2 with i0 < i1 the kept
 *     positions; two groups per byte, the even group in the low nibble.
 *
 * Build: plain C11, no intrinsics, -ffp-contract=off so that every fp32
 * operation rounds on its own on any host ISA.  OpenMP (optional) splits the
 * outer loop over rows only; every output element is computed by one thread
 * in the order written.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define E4M3_MAX_FINITE 448.0

/* ---------------------------------------------------------------- helpers */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
float ora_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Value of an e4m3 code, straight from the format definition. */
double ora_e4m3_to_f64(uint8_t q)
{
    int s = (q >> 7) & 1;
    int e = (q >> 3) & 0xF;
    int m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);           /* subnormal: (m/8) * 2^(1-7) */
    else
        v = ldexp(8.0 + (double)m, e - 10); /* normal: (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Nearest e4m3 code to x: round to nearest, ties to the even code (the code's
 * lowest bit is the mantissa's lowest bit); |x| >= 448 saturates to 448; the
 * sign bit is always copied, so small negatives give -0 (0x80).
 * Finds the bracketing pair of non-negative codes by bisection over the
 * ordered code range 0x00..0x7E, then compares the two distances exactly in
 * double (fp32 inputs and e4m3 values are both exact there). */
uint8_t ora_e4m3_from_f32(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    int lo, hi;
    double dlo, dhi;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    if (a >= E4M3_MAX_FINITE) return (uint8_t)(sign | 0x7E);
    lo = 0x00;  /* value(lo) <= a */
    hi = 0x7E;  /* value(hi) >  a */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (ora_e4m3_to_f64((uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    dlo = a - ora_e4m3_to_f64((uint8_t)lo);
    dhi = ora_e4m3_to_f64((uint8_t)hi) - a;
    if (dlo < dhi) return (uint8_t)(sign | lo);
    if (dhi < dlo) return (uint8_t)(sign | hi);
    return (uint8_t)(sign | ((lo & 1) == 0 ? lo : hi));
}

/* Elementwise ora_e4m3_from_f32 over an array. */
void ora_e4m3_encode_array(const float *x, int64_t n, uint8_t *q)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) q[i] = ora_e4m3_from_f32(x[i]);
}

/* --------------------------------------------------------------- pruning */

/* Kept positions of one group of four bf16 values.  The magnitude of a finite
 * bf16 orders like its bit pattern with the sign cleared (which also makes
 * +0 and -0 equal).  rank_i = number of elements that beat element i, where
 * j beats i if |v_j| > |v_i|, or |v_j| == |v_i| and j < i.  The two elements
 * of rank 0 and 1 are kept; keep[0] < keep[1]. */
void ora_keep2(const uint16_t v[4], int keep[2])
{
    unsigned a[4];
    int i, j, n = 0;
    for (i = 0; i < 4; ++i) a[i] = v[i] & 0x7FFFu;
    for (i = 0; i < 4; ++i) {
        int rank = 0;
        for (j = 0; j < 4; ++j)
            if (a[j] > a[i] || (j < i && a[j] == a[i])) ++rank;
        if (rank < 2) keep[n++] = i;
    }
}

/* Pruned copy of W (bf16 bits): the two dropped positions of every group set
 * to +0.  W is [N][K] with row stride ldw; out is [N][K] packed. */
void ora_prune(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, uint16_t *out)
{
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        int64_t g;
        for (g = 0; g < K / 4; ++g) {
            const uint16_t *v = W + n * ldw + 4 * g;
            int keep[2], i;
            ora_keep2(v, keep);
            for (i = 0; i < 4; ++i)
                out[n * K + 4 * g + i] = (i == keep[0] || i == keep[1]) ? v[i] : 0;
        }
    }
}

/* ---------------------------------------------------------------- scales */

/* Scale of one block: amax over the block (fp32), divided by 448 in fp32;
 * 1 for an all-zero block. */
static float block_scale(const uint16_t *W, int64_t ldw, int64_t r0, int64_t r1,
                         int64_t c0, int64_t c1)
{
    float amax = 0.0f;
    int64_t r, c;
    for (r = r0; r < r1; ++r)
        for (c = c0; c < c1; ++c) {
            float a = fabsf(ora_bf16_to_f32(W[r * ldw + c]));
            if (a > amax) amax = a;
        }
    if (amax == 0.0f) return 1.0f;
    return amax / (float)E4M3_MAX_FINITE;
}

/* Weight scales for granularity (gN, gK): layout [K/gK][ceil(N/gN)], the
 * N-group index fastest (the "M-major" scale layout of CUTLASS PR #2095
 * applied to the weight, which sits in the GEMM's M slot). */
void ora_weight_scales(const uint16_t *W, int64_t N, int64_t K, int64_t ldw,
                       int gN, int gK, float *scales)
{
    int64_t nG = (N + gN - 1) / gN, kB = K / gK, ng;
#pragma omp parallel for schedule(static)
    for (ng = 0; ng < nG; ++ng) {
        int64_t kb;
        int64_t r1 = (ng + 1) * gN < N ? (ng + 1) * gN : N;
        for (kb = 0; kb < kB; ++kb)
            scales[kb * nG + ng] = block_scale(W, ldw, ng * gN, r1, kb * gK, (kb + 1) * gK);
    }
}

/* ----------------------------------------------------------- compression */

/* Prune, scale, quantize and pack.
 *   values[n][K/2]: kept e4m3 codes, two per group, in ascending k;
 *   meta[n][K/8]:   one nibble per group (i0 | i1<<2), group 2j in the low
 *                   nibble of byte j, group 2j+1 in the high nibble;
 *   scales:         as ora_weight_scales.
 * The scale of an element's block is computed from the unpruned W; pruning
 * never removes a group's largest magnitude, so this equals the amax of the
 * pruned block. */
void ora_compress(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, int gN, int gK,
                  uint8_t *values, uint8_t *meta, float *scales)
{
    int64_t nG = (N + gN - 1) / gN, n;
    ora_weight_scales(W, N, K, ldw, gN, gK, scales);
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        int64_t g;
        for (g = 0; g < K / 8; ++g) meta[n * (K / 8) + g] = 0;
        for (g = 0; g < K / 4; ++g) {
            const uint16_t *v = W + n * ldw + 4 * g;
            float s = scales[((4 * g) / gK) * nG + n / gN];
            int keep[2], t;
            ora_keep2(v, keep);
            for (t = 0; t < 2; ++t) {
                float q = ora_bf16_to_f32(v[keep[t]]) / s;
                values[n * (K / 2) + 2 * g + t] = ora_e4m3_from_f32(q);
            }
            meta[n * (K / 8) + g / 2] |= (uint8_t)((keep[0] | (keep[1] << 2)) << (4 * (g & 1)));
        }
    }
}

/* Dense [N][K] e4m3 codes from the packed form; dropped positions are +0. */
void ora_decompress(const uint8_t *values, const uint8_t *meta, int64_t N, int64_t K,
                    uint8_t *dense)
{
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        int64_t g;
        for (g = 0; g < K; ++g) dense[n * K + g] = 0;
        for (g = 0; g < K / 4; ++g) {
            int nib = (meta[n * (K / 8) + g / 2] >> (4 * (g & 1))) & 0xF;
            int i0 = nib & 3, i1 = (nib >> 2) & 3;
            dense[n * K + 4 * g + i0] = values[n * (K / 2) + 2 * g];
            dense[n * K + 4 * g + i1] = values[n * (K / 2) + 2 * g + 1];
        }
    }
}

/* ------------------------------------------------------- storage layout */

/* The packed weight as the C ABI stores it: 128-row x 128-K tiles, each tile
 * contiguous, tiles of one 128-row band consecutive along K.
 *   values: tile t = (n/128)*(K/128) + j/64 holds 128 rows x 64 kept bytes
 *           (8192 B); kept byte j of row n sits at row r = n % 128, byte
 *           b = j % 64, whose 16-byte chunk b/16 is stored at chunk position
 *           (b/16) XOR ((r/2) mod 4) -- the 64-byte swizzle -- so a tile
 *           offset is r*64 + 16*((b/16) ^ ((r/2)%4)) + b%16.
 *   meta:   tile t = (n/128)*(K/128) + jb/16 holds 128 rows x 16 bytes
 *           (2048 B); logical meta byte jb of row n sits at r*16 + jb%16.
 * N must be a multiple of 128 and K of 128. */
static int64_t values_tiled_offset(int64_t n, int64_t j, int64_t K)
{
    int64_t t = (n / 128) * (K / 128) + j / 64;
    int64_t r = n % 128, b = j % 64;
    return t * 8192 + r * 64 + 16 * ((b / 16) ^ ((r / 2) % 4)) + b % 16;
}

static int64_t meta_tiled_offset(int64_t n, int64_t jb, int64_t K)
{
    int64_t t = (n / 128) * (K / 128) + jb / 16;
    return t * 2048 + (n % 128) * 16 + jb % 16;
}

void ora_tile_values(const uint8_t *values, int64_t N, int64_t K, uint8_t *tiled)
{
    int64_t n, j;
    for (n = 0; n < N; ++n)
        for (j = 0; j < K / 2; ++j) tiled[values_tiled_offset(n, j, K)] = values[n * (K / 2) + j];
}

void ora_untile_values(const uint8_t *tiled, int64_t N, int64_t K, uint8_t *values)
{
    int64_t n, j;
    for (n = 0; n < N; ++n)
        for (j = 0; j < K / 2; ++j) values[n * (K / 2) + j] = tiled[values_tiled_offset(n, j, K)];
}

void ora_tile_meta(const uint8_t *meta, int64_t N, int64_t K, uint8_t *tiled)
{
    int64_t n, jb;
    for (n = 0; n < N; ++n)
        for (jb = 0; jb < K / 8; ++jb) tiled[meta_tiled_offset(n, jb, K)] = meta[n * (K / 8) + jb];
}

void ora_untile_meta(const uint8_t *tiled, int64_t N, int64_t K, uint8_t *meta)
{
    int64_t n, jb;
    for (n = 0; n < N; ++n)
        for (jb = 0; jb < K / 8; ++jb) meta[n * (K / 8) + jb] = tiled[meta_tiled_offset(n, jb, K)];
}

/* ------------------------------------------------- activation quantization */

/* Dynamic activation quantization (pytorch/ao PR #3258, the activation path:
 * divide by the scale, then cast to e4m3).  X fp32 [M][K] (row stride ldx);
 * one scale per token and K block of length gK: sx[K/gK][M], M fastest;
 * sx = amax/448 (1 for an all-zero block); xq[m][k] = e4m3(x / sx). */
void ora_quantize_act(const float *X, int64_t M, int64_t K, int64_t ldx, int gK,
                      uint8_t *xq, float *sx)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int64_t kb, k;
        for (kb = 0; kb < K / gK; ++kb) {
            float amax = 0.0f, s;
            for (k = kb * gK; k < (kb + 1) * gK; ++k) {
                float a = fabsf(X[m * ldx + k]);
                if (a > amax) amax = a;
            }
            s = amax == 0.0f ? 1.0f : amax / (float)E4M3_MAX_FINITE;
            sx[kb * M + m] = s;
            for (k = kb * gK; k < (kb + 1) * gK; ++k)
                xq[m * K + k] = ora_e4m3_from_f32(X[m * ldx + k] / s);
        }
    }
}

/* ------------------------------------------------------------------- GEMM */

/* Group-wise scaled sparse GEMM, Y[m][n] for every token m and channel n:
 *   for each K block kb of length gK (kb ascending):
 *       P  = sum over kept k in the block, k ascending, of wq[n][k] * xq[m][k]
 *       acc = acc + (sx[kb][m/gM] * sw[kb][n/gN]) * P
 *   acc = acc + sum_{j<r} X2[m][j] * W2[n][j]          (bf16 side GEMM)
 *   acc = acc + bias[n]                                (bf16 bias, if any)
 * The bias is that of the linear operation of pytorch/ao PR #3258
 * (input, weight, bias), added last, before the output is rounded.
 * Only kept weights are multiplied (the sparse loop); wq comes from values
 * and the metadata nibbles.  Every product of two e4m3 values, and of two
 * bf16 values, is exact in fp32.  acc_fp64 = 0 accumulates in fp32 (each
 * operation rounded, as written above); 1 accumulates in double.
 * Layouts: xq [M][K] row stride ldx; sx [K/gK][ceil(M/gM)]; values [N][K/2];
 * meta [N][K/8]; sw [K/gK][ceil(N/gN)]; X2 [M][r]; W2 [N][r]; bias [N] or
 * NULL; Y [M][N]. */
void ora_gemm(const uint8_t *xq, const float *sx, int64_t M, int64_t K, int64_t ldx, int gM,
              const uint8_t *values, const uint8_t *meta, const float *sw, int64_t N,
              int gN, int gK, const uint16_t *X2, const uint16_t *W2, int64_t r,
              const uint16_t *bias, int acc_fp64, double *Y)
{
    int64_t ldsx = (M + gM - 1) / gM, ldsw = (N + gN - 1) / gN, kB = K / gK;
    double dec[256];
    int64_t m;
    int i;
    for (i = 0; i < 256; ++i) dec[i] = ora_e4m3_to_f64((uint8_t)i);
#pragma omp parallel for schedule(dynamic, 1)
    for (m = 0; m < M; ++m) {
        int64_t n;
        for (n = 0; n < N; ++n) {
            float accf = 0.0f;
            double accd = 0.0;
            int64_t kb, g, j;
            for (kb = 0; kb < kB; ++kb) {
                float pf = 0.0f;
                double pd = 0.0;
                for (g = kb * gK / 4; g < (kb + 1) * gK / 4; ++g) {
                    int nib = (meta[n * (K / 8) + g / 2] >> (4 * (g & 1))) & 0xF;
                    int i0 = nib & 3, i1 = (nib >> 2) & 3;
                    double p0 = dec[values[n * (K / 2) + 2 * g]] * dec[xq[m * ldx + 4 * g + i0]];
                    double p1 = dec[values[n * (K / 2) + 2 * g + 1]] * dec[xq[m * ldx + 4 * g + i1]];
                    if (acc_fp64) { pd += p0; pd += p1; }
                    else { pf += (float)p0; pf += (float)p1; }
                }
                if (acc_fp64) {
                    accd += ((double)sx[kb * ldsx + m / gM] * (double)sw[kb * ldsw + n / gN]) * pd;
                } else {
                    float s = sx[kb * ldsx + m / gM] * sw[kb * ldsw + n / gN];
                    accf += s * pf;
                }
            }
            for (j = 0; j < r; ++j) {
                double p = (double)ora_bf16_to_f32(X2[m * r + j]) * (double)ora_bf16_to_f32(W2[n * r + j]);
                if (acc_fp64) accd += p; else accf += (float)p;
            }
            if (bias) {
                float b = ora_bf16_to_f32(bias[n]);
                if (acc_fp64) accd += (double)b; else accf += b;
            }
            Y[m * N + n] = acc_fp64 ? accd : (double)accf;
        }
    }
}

/* ------------------------------------------------------------ int8 sibling */

/* The int8 x int8 2:4 sibling of the FP8 path.  pytorch/ao PR #3258 (review:
 * the only 2:4 kernels are int8 x int8 and fp8 x fp8; Int8SemiSparseTensor)
 * names it but defines no int8 quantizer, so the plainest symmetric one is
 * taken:
 *   - scale = amax / 127 (fp32, correctly rounded) per output channel for
 *     the weight and per token for the activation; 1 for an all-zero row;
 *   - q = the integer nearest to the correctly rounded fp32 quotient x/scale,
 *     ties to even, clamped to [-127, 127] (|x| <= amax keeps it inside);
 *   - pruning, metadata and storage as for the FP8 weight, one byte (two's
 *     complement) per kept value;
 *   - GEMM: acc = the exact integer sum of the kept products, then
 *     y = (sx * sw) * float(acc) in fp32, plus the bf16 bias if any. */
#define INT8_MAX_Q 127.0f

/* Nearest integer, ties to even, written out (no dependence on the host's
 * rounding mode): x - floor(x) is exact for |x| < 2^23. */
static float round_half_even(float x)
{
    float f = floorf(x), d = x - f;
    if (d > 0.5f) return f + 1.0f;
    if (d < 0.5f) return f;
    return fmodf(f, 2.0f) == 0.0f ? f : f + 1.0f;
}

int8_t ora_int8_from_f32(float x)
{
    float r = round_half_even(x);
    if (r > INT8_MAX_Q) r = INT8_MAX_Q;
    if (r < -INT8_MAX_Q) r = -INT8_MAX_Q;
    return (int8_t)r;
}

static float int8_scale(float amax)
{
    return amax == 0.0f ? 1.0f : amax / INT8_MAX_Q;
}

/* values[n][K/2] int8 (as bytes), meta[n][K/8] as ora_compress, scales[n]. */
void ora_compress_int8(const uint16_t *W, int64_t N, int64_t K, int64_t ldw,
                       uint8_t *values, uint8_t *meta, float *scales)
{
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        int64_t g, k;
        float amax = 0.0f, s;
        for (k = 0; k < K; ++k) {
            float a = fabsf(ora_bf16_to_f32(W[n * ldw + k]));
            if (a > amax) amax = a;
        }
        s = int8_scale(amax);
        scales[n] = s;
        for (g = 0; g < K / 8; ++g) meta[n * (K / 8) + g] = 0;
        for (g = 0; g < K / 4; ++g) {
            const uint16_t *v = W + n * ldw + 4 * g;
            int keep[2], t;
            ora_keep2(v, keep);
            for (t = 0; t < 2; ++t)
                values[n * (K / 2) + 2 * g + t] = (uint8_t)ora_int8_from_f32(ora_bf16_to_f32(v[keep[t]]) / s);
            meta[n * (K / 8) + g / 2] |= (uint8_t)((keep[0] | (keep[1] << 2)) << (4 * (g & 1)));
        }
    }
}

/* Per-token int8 quantization of X fp32 [M][K] (row stride ldx): xq [M][K]
 * int8 (as bytes), sx [M]. */
void ora_quantize_act_int8(const float *X, int64_t M, int64_t K, int64_t ldx, uint8_t *xq, float *sx)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int64_t k;
        float amax = 0.0f, s;
        for (k = 0; k < K; ++k) {
            float a = fabsf(X[m * ldx + k]);
            if (a > amax) amax = a;
        }
        s = int8_scale(amax);
        sx[m] = s;
        for (k = 0; k < K; ++k) xq[m * K + k] = (uint8_t)ora_int8_from_f32(X[m * ldx + k] / s);
    }
}

/* Y[m][n] = (sx[m] * sw[n]) * float(acc[m][n]) (+ bias[n]) with acc the exact
 * integer sum over the kept k of wq[n][k] * xq[m][k].  acc [M][N] (int32, or
 * NULL) receives the sums; K <= 131072 keeps them inside int32. */
void ora_gemm_int8(const uint8_t *xq, const float *sx, int64_t M, int64_t K, int64_t ldx,
                   const uint8_t *values, const uint8_t *meta, const float *sw, int64_t N,
                   const uint16_t *bias, int32_t *acc, double *Y)
{
    int64_t m;
#pragma omp parallel for schedule(dynamic, 1)
    for (m = 0; m < M; ++m) {
        int64_t n;
        for (n = 0; n < N; ++n) {
            int64_t a = 0, g;
            float y;
            for (g = 0; g < K / 4; ++g) {
                int nib = (meta[n * (K / 8) + g / 2] >> (4 * (g & 1))) & 0xF;
                int i0 = nib & 3, i1 = (nib >> 2) & 3;
                a += (int64_t)(int8_t)values[n * (K / 2) + 2 * g] * (int8_t)xq[m * ldx + 4 * g + i0];
                a += (int64_t)(int8_t)values[n * (K / 2) + 2 * g + 1] * (int8_t)xq[m * ldx + 4 * g + i1];
            }
            if (acc) acc[m * N + n] = (int32_t)a;
            y = (sx[m] * sw[n]) * (float)a;
            if (bias) y += ora_bf16_to_f32(bias[n]);
            Y[m * N + n] = (double)y;
        }
    }
}

/* Threads the OpenMP loops above use (1 without OpenMP). */
int ora_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
