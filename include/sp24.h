/*
 * sp24.h -- C ABI of libsp24: 2:4 semi-structured sparse FP8 (e4m3) linear
 * layer on a GB300 (sm_103a).
 *
 *   Y[M,N] (bf16) = X[M,K] . W[N,K]^T  with W pruned 2:4 along K,
 *   both operands e4m3 with group-wise fp32 scales, plus an optional bf16
 *   side term X2[M,r] . W2[N,r]^T added into the same output.
 *
 * General conventions
 *   - Pointers marked (device) are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or retains them.  Pointers marked
 *     (host) are ordinary host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is stream-ordered and asynchronous; none
 *     synchronises except sp24_last_device_error().
 *   - Every entry point checks its arguments before launching anything and
 *     returns an sp24_status; nothing throws across the ABI.  On an error
 *     no kernel has been launched and no output has been written.
 *   - Row-major storage; "ld" arguments are row strides in elements.
 *   - Scale tensors use the layout [K/gK][ceil(rows/g)] with the row-group
 *     index fastest (the "M-major" scale layout of CUTLASS PR #2095,
 *     "Improvements for: Groupwise scaling along M for FP8 gemm", PR
 *     description).  gK = K means one block along K.
 *
 * The pages this follows are cited by title and comment thread:
 *   [2029] CUTLASS issue #2029, "[QST] CUTLASS support for fp8 sparse
 *          matrix(for W) multiplication ... sparse tensor core";
 *   [2095] CUTLASS PR #2095, "Improvements for: Groupwise scaling along M
 *          for FP8 gemm";
 *   [2058] CUTLASS issue #2058, "[QST] How to implement a fused mixed
 *          precision matrix multiplication such as w4a4 + w16a16?";
 *   [3258] pytorch/ao PR #3258, "Introduce new W8A8-FP-CSR quantization API".
 */
#ifndef SP24_H
#define SP24_H

#include <stddef.h>
#include <stdint.h>

#if defined(SP24_BUILD) && defined(__GNUC__)
#define SP24_API __attribute__((visibility("default")))
#else
#define SP24_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SP24_OK = 0,
  SP24_ERR_INVALID_ARG = 1,    /* null pointer, bad size or stride            */
  SP24_ERR_UNSUPPORTED = 2,    /* valid but not implemented (granularity ...) */
  SP24_ERR_ALIGNMENT = 3,      /* pointer or row stride not 16-byte aligned   */
  SP24_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed           */
  SP24_ERR_ARCH = 5,           /* current device is not sm_103                */
  SP24_ERR_WORKSPACE = 6,      /* workspace missing or too small              */
  SP24_ERR_DEVICE_TIMEOUT = 7  /* a kernel gave up waiting (device error word)*/
} sp24_status;

/* Human-readable name of a status code (static string). */
SP24_API const char* sp24_status_string(sp24_status s);

/* Bytes of sparsity metadata for an N x K weight: N * K / 8 (one 4-bit
 * entry per group of four along K).  K must be a multiple of 8. */
SP24_API size_t sp24_meta_bytes(int64_t N, int64_t K);

/*
 * sp24_fp8_compress -- magnitude 2:4 prune + e4m3 quantize + pack.
 * Follows [3258] (jcaip's review: drop the two smallest |w| of each group of
 * four along K; positive amax-based scales; keep only the specified values
 * and the sparsity metadata, nothing dense; an all-zero weight is legal) and
 * [2095] for the 128x128 block scale granularity.
 *
 *   W       (device) bf16 [N][K], row stride ldw >= K elements.
 *   gN, gK  weight scale granularity: (1, K) per output channel,
 *           (1, 128) per channel and 128-wide K block, or (128, 128) blocks.
 *   values  (device, out) N*K/2 bytes of kept e4m3 codes in tiled storage:
 *           the weight is cut into 128-row x 128-K tiles; tile
 *           t = (n/128)*(K/128) + k/128 occupies bytes [8192 t, 8192 t + 8192).
 *           Inside a tile, row r = n % 128 owns 64 bytes at 64 r: the two kept
 *           codes of each group of four, in ascending k (kept index j = 2g + t
 *           for group g), with the 16-byte chunk c = (j % 64) / 16 stored at
 *           chunk position c XOR ((r / 2) mod 4) (the 64-byte swizzle the
 *           tensor core reads).  A whole tile is one contiguous copy.
 *   meta    (device, out) sp24_meta_bytes(N, K) = N*K/8 bytes, tiled the same
 *           way: tile t occupies [2048 t, 2048 t + 2048); row r owns 16 bytes
 *           at 16 r; byte b carries group 2b of the tile row in its low nibble
 *           and group 2b+1 in its high nibble; a nibble is i0 | (i1 << 2),
 *           i0 < i1 the kept positions within the group.  This is the layout
 *           the tensor core's sparse metadata takes in tensor memory (lane =
 *           row), so the GEMM copies it without rearranging.
 *   scales  (device, out) fp32 [K/gK][ceil(N/gN)]: amax/448 of the block
 *           (1.0 for an all-zero block).
 * Each kept element is q = e4m3_rn_satfinite(w / scale) with a correctly
 * rounded fp32 division.  Ties in |w| keep the lower index.
 * Preconditions: N a positive multiple of 128; K a positive multiple of 128;
 * W, values and meta 16-byte aligned, ldw*2 a multiple of 16.
 */
SP24_API sp24_status sp24_fp8_compress(const void* W, int64_t N, int64_t K, int64_t ldw, int gN, int gK,
                              void* values, void* meta, float* scales, void* stream);

/*
 * sp24_fp8_decompress -- the dense dequantized weight from the compressed
 * storage: W[n][k] = bf16(sw[k/gK][n/gN] * decode(value)) at the two kept
 * positions of every group of four along K, +0 at the other two.  It is what
 * sp24_fp8_gemm returns for an identity activation with unit scales ([3258],
 * jcaip's review: dequantize by multiplying with an identity), computed
 * directly: the product is rounded to fp32, then to bf16.
 *
 *   values, meta, scales (device) as produced by sp24_fp8_compress for [N][K]
 *           with granularities gN, gK (the same combinations).
 *   W       (device, out) bf16 [N][K], row stride ldw >= K, ldw*2 a multiple
 *           of 16, 16-byte aligned.
 * Preconditions: N a positive multiple of 128; K a positive multiple of 128.
 */
SP24_API sp24_status sp24_fp8_decompress(const void* values, const void* meta, const float* scales, int64_t N,
                                int64_t K, int gN, int gK, void* W, int64_t ldw, void* stream);

/*
 * sp24_fp8_quantize_act -- dynamic activation quantization to e4m3.
 * Follows [3258] (the activation path divides by the scale, then casts to
 * e4m3) with the per-token / 1x128 granularities of [2095].
 *
 *   X   (device) fp32 [M][K], row stride ldx >= K.
 *   gK  K or 128 (scales per token, or per token and 128-wide K block).
 *   xq  (device, out) uint8 e4m3 [M][K] (row stride K).
 *   sx  (device, out) fp32 [K/gK][M]: amax/448 (1.0 for an all-zero block).
 * Preconditions: M >= 1; K a positive multiple of 128; X and xq 16-byte
 * aligned; ldx*4 a multiple of 16.
 */
SP24_API sp24_status sp24_fp8_quantize_act(const float* X, int64_t M, int64_t K, int64_t ldx, int gK, void* xq,
                                  float* sx, void* stream);

/*
 * sp24_fp8_quantize_act_bf16 -- the same for bf16 activations (the dtype of
 * the bf16 models the pages quantize): X (device) bf16 [M][K], row stride
 * ldx >= K with ldx*2 a multiple of 16.  Every bf16 value is an fp32 value,
 * so the result is that of sp24_fp8_quantize_act on X widened to fp32.
 */
SP24_API sp24_status sp24_fp8_quantize_act_bf16(const void* X, int64_t M, int64_t K, int64_t ldx, int gK, void* xq,
                                       float* sx, void* stream);

/*
 * sp24_fp8_gemm -- group-wise scaled 2:4 sparse FP8 GEMM with an optional
 * fused bf16 side GEMM:
 *
 *   Y[m][n] = bf16( sum_kb sx[kb][m/gM] * sw[kb][n/gN] * P_kb[m][n]
 *                   + sum_{j<r} X2[m][j] * W2[n][j] + bias[n] )
 *   P_kb[m][n] = sum over k in K block kb of xq[m][k] * wq[n][k]  (fp32)
 *
 * where wq is the dense weight that (values, meta) encode.  Internally the
 * product is computed as Y^T = W . X^T so that the sparse weight is the
 * row-major sparse A operand of the tensor core ([2029], klevzoff's
 * swap+transpose answer); no data is moved for that.  Per-K-block partial
 * sums are scaled and added to the running fp32 sum ([2095], promotion per K
 * tile).  Token rows beyond M in the last tile are computed on zero fill and
 * not stored ([2095], predication of partial tiles).  The side GEMM is the
 * small w16a16 term of [2058] (hyx1999: Y = X1 W1^T + X2 W2^T in one kernel).
 * The bias is that of the linear operation in [3258]
 * (_linear_fp8_act_fp8_weight_sparse_cutlass_impl(input, weight, bias)),
 * added in fp32 before the one rounding to bf16.
 *
 *   Xq      (device) uint8 e4m3 [M][K], row stride ldx (ldx % 16 == 0).
 *   sx      (device) fp32 [K/gK][ceil(M/gM)].
 *   gM      1 or 128.
 *   values, meta (device) as produced by sp24_fp8_compress for [N][K].
 *   sw      (device) fp32 [K/gK][ceil(N/gN)].
 *   gN      1 or 128; gK: K or 128.
 *   X2, W2  (device) bf16 [M][r] and [N][r] (row stride r), or NULL with
 *           r = 0 for no side GEMM; r a multiple of 16, at most 64.
 *   bias    (device) bf16 [N], 2-byte aligned, or NULL for none.
 *   Y       (device, out) bf16 [M][N], row stride ldy >= N, ldy % 8 == 0,
 *           16-byte aligned.
 *   workspace, workspace_bytes: device scratch of at least
 *           sp24_fp8_gemm_workspace_size(M, N, K, r) bytes, 16-byte aligned
 *           (may be NULL when that size is 0).  Only the stream-K
 *           decomposition of small-token calls uses it (see
 *           sp24_set_decomposition; the size is 0 for the others): the launch
 *           deals the (tile, K block) work out to one CTA per SM in equal
 *           contiguous ranges, and a tile cut between CTAs is finished by the
 *           CTA holding its first K blocks, which adds the others' fp32
 *           partials in a fixed order (the result does not depend on
 *           timing).  The workspace holds a launch counter, one
 *           flag per CTA and one partial tile per CTA.  Zero it once before
 *           its first use; each launch leaves it consistent for the next,
 *           whatever the shape, CUDA graph replays included, and a launch
 *           that gave up on a wait (SP24_ERR_DEVICE_TIMEOUT) as well: every
 *           CTA counts itself out of the launch counter before it exits.
 *           Calls that overlap on the GPU must not share it.  With less than the
 *           queried size the call runs with whole tiles per CTA.
 * Preconditions: M >= 1; N a positive multiple of 128; K a positive multiple
 * of 128; all scales finite and > 0; device pointers 16-byte aligned.
 * Errors: SP24_ERR_* as above; device-side wait timeouts are reported by
 * sp24_last_device_error().
 */
SP24_API sp24_status sp24_fp8_gemm(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx, int gM,
                          const void* values, const void* meta, const float* sw, int64_t N, int gN, int gK,
                          const void* X2, const void* W2, int64_t r, const void* bias, void* Y, int64_t ldy,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * sp24_fp8_gemm_batched -- L independent problems of one shape in one call:
 * Y_l = sp24_fp8_gemm(Xq_l, sx_l, values_l, meta_l, sw_l, bias_l) for
 * l < L, with problem l's operands at base + l * stride (the batched L mode
 * of CUTLASS's (M, N, K, L) problem shape, [2095]).  No side GEMM.
 *
 *   stride_x, stride_values, stride_meta: bytes between problems (multiples
 *           of 16; Xq, values and meta of one problem at least M*ldx,
 *           N*K/2 and N*K/8 bytes);
 *   stride_sx, stride_sw, stride_bias, stride_y: elements between problems
 *           (fp32, fp32, bf16, bf16; stride_y*2 a multiple of 16).
 *   workspace: L times the single problem's sp24_fp8_gemm_workspace_size
 *           for stream-K, zeroed before its first use as for sp24_fp8_gemm
 *           (less: whole tiles per CTA).
 * Problems small enough to leave SMs idle run in one launch whose persistent
 * CTAs take work units from every problem; problems that fill the GPU on
 * their own (the SM-pair cases) run as back-to-back launches.
 */
SP24_API sp24_status sp24_fp8_gemm_batched(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx, int gM,
                                  const void* values, const void* meta, const float* sw, int64_t N, int gN, int gK,
                                  const void* bias, void* Y, int64_t ldy, int64_t L, int64_t stride_x,
                                  int64_t stride_sx, int64_t stride_values, int64_t stride_meta, int64_t stride_sw,
                                  int64_t stride_bias, int64_t stride_y, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * sp24_fp8_gemm_fixed_scratch -- sp24_fp8_gemm for callers that may not
 * allocate.  The pages have no counterpart to this entry point.
 *
 * Some callers own their device memory outright and must not allocate while
 * they run (serving loops that plan every buffer at start-up, code hosted in
 * a framework whose allocator this library cannot reach).  This call takes
 * the same arguments as sp24_fp8_gemm minus the workspace and computes the
 * same result; the stream-K scratch comes from a fixed 8 MiB array inside the
 * library's device image instead.  It calls no allocating routine.
 *   - Every GPU that loads the library holds that array until the process
 *     exits, and all calls on a device share it: calls that overlap on the
 *     GPU (other streams, other host threads) race on it and corrupt each
 *     other's results.  Serialise them.
 *   - Every call looks up the array's device address in the current
 *     device's context (so a context that was reset and created again gets
 *     the new address).  The first call on a device may load the library's
 *     device image there; make that first call before any stream capture.
 *   - A shape whose scratch need (sp24_fp8_gemm_workspace_size) exceeds
 *     8 MiB is refused with SP24_ERR_WORKSPACE.  No shape needs that much
 *     on parts with up to 240 SMs (the 152-SM GB300 among them): the refusal
 *     guards larger parts.  Shapes that need no scratch always run.
 * The array starts zeroed, and the stream-K counter and flags keep it
 * consistent from call to call.  That holds after SP24_ERR_DEVICE_TIMEOUT
 * too: a launch that gave up on a wait still counts every CTA out of the
 * counter, so nothing is left for the caller to reset.
 */
SP24_API sp24_status sp24_fp8_gemm_fixed_scratch(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx,
                                                 int gM, const void* values, const void* meta, const float* sw,
                                                 int64_t N, int gN, int gK, const void* X2, const void* W2, int64_t r,
                                                 const void* bias, void* Y, int64_t ldy, void* stream);

/* Device scratch bytes sp24_fp8_gemm needs for this problem (0 = none). */
SP24_API size_t sp24_fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int64_t r);

/*
 * sp24_set_decomposition -- how later GEMM calls of this process deal out
 * the tiles' K ranges (CUTLASS's stream-K decomposition modes, [2095]'s
 * kernel schedules).  Process-wide; sp24_fp8_gemm_workspace_size answers for
 * the mode in force, so query it after setting the mode.
 *   SP24_DECOMP_HEURISTIC     (default) whichever of the three below the
 *                             library's cost model expects to be fastest;
 *   SP24_DECOMP_DATA_PARALLEL whole tiles only (no workspace needed);
 *   SP24_DECOMP_STREAM_K      stream-K wherever it applies: all tiles' K
 *                             stages dealt out to one CTA per SM, partials
 *                             exchanged through the workspace;
 *   SP24_DECOMP_CLUSTER_SPLIT each tile's K range split across the CTAs of a
 *                             thread-block cluster (4 CTAs, or 2 when 4 do
 *                             not fit or for 33 to 64 tokens), partials
 *                             reduced through
 *                             distributed shared memory (no workspace), when
 *                             every tile's cluster fits on the SMs at once.
 * Both splits apply to per-tensor-K scaling without a side GEMM and at most
 * 64 tokens (the one-SM kernel's small-token tiles), when a tile's K range
 * spans at least two pipeline stages (a stage holds up to four 128-wide K
 * blocks for up to 32 tokens, two above); other calls ignore the mode.
 * Results are the same within rounding (each mode has a fixed summation
 * order, so each is deterministic).
 * Errors: SP24_ERR_INVALID_ARG for an unknown mode.
 */
enum {
  SP24_DECOMP_HEURISTIC = 0,
  SP24_DECOMP_DATA_PARALLEL = 1,
  SP24_DECOMP_STREAM_K = 2,
  SP24_DECOMP_CLUSTER_SPLIT = 3
};
SP24_API sp24_status sp24_set_decomposition(int mode);

/*
 * sp24_fp8_gemm_decomposition -- the decomposition a call of this shape
 * with per-tensor-K scaling would use under the mode in force:
 * SP24_DECOMP_DATA_PARALLEL, SP24_DECOMP_STREAM_K or
 * SP24_DECOMP_CLUSTER_SPLIT (and, if cluster_size is not NULL, the CTAs
 * per tile there, else 1).  Returns -1 for an invalid shape or without a
 * usable device.  Stream-K also needs the workspace; without it the call
 * runs whole tiles.
 */
SP24_API int sp24_fp8_gemm_decomposition(int64_t M, int64_t N, int64_t K, int64_t r, int* cluster_size);

/*
 * sp24_last_device_error -- synchronise `stream`, then read and clear the
 * library's device error word on the current device.  Returns SP24_OK, or
 * SP24_ERR_DEVICE_TIMEOUT if any kernel of this library gave up on a bounded
 * wait since the last call (its results are then invalid), or SP24_ERR_CUDA.
 */
SP24_API sp24_status sp24_last_device_error(void* stream);

/*
 * ---------------------------------------------------------- int8 sibling
 * The int8 x int8 2:4 path ([3258], review: the 2:4 kernels are int8 x int8
 * and fp8 x fp8; Int8SemiSparseTensor).  The pages name it but give no int8
 * quantizer; the plain symmetric one is used: scale = amax / 127 (correctly
 * rounded fp32; 1.0 for an all-zero row), code = the integer nearest to the
 * correctly rounded quotient x / scale, ties to even, in [-127, 127].
 *
 * sp24_int8_compress -- magnitude 2:4 pruning along K (as sp24_fp8_compress),
 * int8 codes with one scale per output channel.
 *   W       (device) bf16 [N][K], row stride ldw >= K (ldw*2 a multiple of 16).
 *   values  (device, out) [N*K/2] int8 codes, meta (device, out) [N*K/8]: the
 *           tiled storage of sp24_fp8_compress, with int8 codes in place of
 *           e4m3 ones.
 *   scales  (device, out) fp32 [N].
 * Preconditions: N a positive multiple of 128; K a positive multiple of 128;
 * W, values, meta 16-byte aligned.
 */
SP24_API sp24_status sp24_int8_compress(const void* W, int64_t N, int64_t K, int64_t ldw, void* values, void* meta,
                               float* scales, void* stream);

/*
 * sp24_int8_quantize_act -- per-token int8 activation quantization.
 *   X   (device) fp32 [M][K], row stride ldx >= K (ldx*4 a multiple of 16).
 *   xq  (device, out) int8 [M][K] (row stride K); sx (device, out) fp32 [M].
 * Preconditions: M >= 1; K a positive multiple of 128; X, xq 16-byte aligned.
 */
SP24_API sp24_status sp24_int8_quantize_act(const float* X, int64_t M, int64_t K, int64_t ldx, void* xq, float* sx,
                                   void* stream);

/*
 * sp24_int8_gemm -- Y[m][n] = bf16( (sx[m] * sw[n]) * float(acc[m][n]) + bias[n] ),
 * acc[m][n] = the exact integer sum over the kept k of wq[n][k] * xq[m][k].
 * Each step is rounded as written (fp32, then bf16 round to nearest even).
 * sm_103a has no int8 tensor-core MMA of the tcgen05 family, so this runs on
 * the warp-level sparse MMA (mma.sp m16n8k64 s8).
 *   Xq  (device) int8 [M][K], row stride ldx >= K (a multiple of 16).
 *   sx  (device) fp32 [M]; values, meta (device) from sp24_int8_compress;
 *   sw  (device) fp32 [N]; bias (device) bf16 [N] or NULL.
 *   Y   (device, out) bf16 [M][N], row stride ldy >= N.
 * Preconditions: M >= 1; N a positive multiple of 128; K a positive multiple
 * of 128 and at most 131072 (SP24_ERR_UNSUPPORTED above: the int32 sums stay
 * exact); Xq, values, meta 16-byte aligned; sx, sw 4-byte aligned.
 */
SP24_API sp24_status sp24_int8_gemm(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx,
                           const void* values, const void* meta, const float* sw, int64_t N, const void* bias,
                           void* Y, int64_t ldy, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SP24_H */
