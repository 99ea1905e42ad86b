"""CPU oracle for the 2:4 sparse FP8 path and its int8 sibling (numpy front end
to ``sp24_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path (``semi_structured_sparse_gb300``) and never imports it.

Every function cites the passage it follows; ``sp24_oracle.c`` holds the
step-by-step definitions.  Arrays are numpy: bf16 tensors travel as their
``uint16`` bit patterns, e4m3 tensors as ``uint8`` codes.
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        L.ora_e4m3_from_f32.argtypes = [ctypes.c_float]
        L.ora_e4m3_from_f32.restype = ctypes.c_uint8
        L.ora_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.ora_e4m3_to_f64.restype = ctypes.c_double
        L.ora_e4m3_encode_array.argtypes = [P, I64, P]
        L.ora_keep2.argtypes = [P, P]
        L.ora_prune.argtypes = [P, I64, I64, I64, P]
        L.ora_weight_scales.argtypes = [P, I64, I64, I64, I, I, P]
        L.ora_compress.argtypes = [P, I64, I64, I64, I, I, P, P, P]
        L.ora_decompress.argtypes = [P, P, I64, I64, P]
        L.ora_quantize_act.argtypes = [P, I64, I64, I64, I, P, P]
        L.ora_gemm.argtypes = [P, P, I64, I64, I64, I, P, P, P, I64, I, I,
                               P, P, I64, P, I, P]
        for f in ("ora_tile_values", "ora_untile_values", "ora_tile_meta", "ora_untile_meta"):
            getattr(L, f).argtypes = [P, I64, I64, P]
        L.ora_num_threads.restype = ctypes.c_int
        L.ora_int8_from_f32.argtypes = [ctypes.c_float]
        L.ora_int8_from_f32.restype = ctypes.c_int8
        L.ora_compress_int8.argtypes = [P, I64, I64, I64, P, P, P]
        L.ora_quantize_act_int8.argtypes = [P, I64, I64, I64, P, P]
        L.ora_gemm_int8.argtypes = [P, P, I64, I64, I64, P, P, P, I64, P, P, P]
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(lib().ora_num_threads())


# ----------------------------------------------------------------- e4m3 codec
def e4m3_encode(x) -> np.ndarray:
    """RNE + satfinite fp32 -> e4m3 codes (OCP E4M3, the float8_e4m3fn type of
    torchao PR #3258).  Output has the input's shape."""
    x = _c(x, np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    lib().ora_e4m3_encode_array(_p(x), x.size, _p(q))
    return q


def e4m3_decode(q) -> np.ndarray:
    """e4m3 codes -> exact float64 values (NaN for S.1111.111)."""
    q = _c(q, np.uint8)
    table = np.array([lib().ora_e4m3_to_f64(i) for i in range(256)], dtype=np.float64)
    return table[q]


# -------------------------------------------------------------------- prune
def keep2(group) -> tuple:
    """Kept positions (i0 < i1) of one group of four bf16 bit patterns
    (torchao PR #3258, jcaip's review: drop the two smallest |w| of each 4)."""
    v = _c(group, np.uint16)
    out = np.zeros(2, dtype=np.int32)
    lib().ora_keep2(_p(v), _p(out))
    return int(out[0]), int(out[1])


def prune(W_bits: np.ndarray) -> np.ndarray:
    """Pruned copy of W (bf16 bits [N,K]); dropped positions set to +0."""
    W = _c(W_bits, np.uint16)
    N, K = W.shape
    out = np.empty_like(W)
    lib().ora_prune(_p(W), N, K, K, _p(out))
    return out


# ------------------------------------------------------------------- scales
def weight_scales(W_bits, gN: int, gK: int) -> np.ndarray:
    """amax/448 per (gN x gK) block, layout [K/gK][ceil(N/gN)]."""
    W = _c(W_bits, np.uint16)
    N, K = W.shape
    nG = (N + gN - 1) // gN
    s = np.empty((K // gK, nG), dtype=np.float32)
    lib().ora_weight_scales(_p(W), N, K, K, gN, gK, _p(s))
    return s


# ------------------------------------------------------------------ compress
def compress(W_bits, gN: int = 1, gK: int = None):
    """Prune + scale + e4m3 + pack (logical metadata layout).

    Returns (values uint8 [N,K/2], meta uint8 [N,K/8], scales fp32 [K/gK,ceil(N/gN)]).
    """
    W = _c(W_bits, np.uint16)
    N, K = W.shape
    gK = K if gK is None else gK
    nG = (N + gN - 1) // gN
    values = np.empty((N, K // 2), dtype=np.uint8)
    meta = np.empty((N, K // 8), dtype=np.uint8)
    scales = np.empty((K // gK, nG), dtype=np.float32)
    lib().ora_compress(_p(W), N, K, K, gN, gK, _p(values), _p(meta), _p(scales))
    return values, meta, scales


def decompress(values, meta) -> np.ndarray:
    """Dense e4m3 codes [N,K] from (values, meta); dropped positions are 0x00."""
    values = _c(values, np.uint8)
    meta = _c(meta, np.uint8)
    N = values.shape[0]
    K = values.shape[1] * 2
    dense = np.empty((N, K), dtype=np.uint8)
    lib().ora_decompress(_p(values), _p(meta), N, K, _p(dense))
    return dense


# ----------------------------------------------------------- storage layout
def tile_values(values) -> np.ndarray:
    """Logical kept values [N, K/2] -> the ABI's tiled storage (N*K/2 bytes):
    contiguous 128-row x 64-byte tiles with the 64-byte swizzle inside."""
    values = _c(values, np.uint8)
    N, K = values.shape[0], values.shape[1] * 2
    out = np.empty(N * K // 2, dtype=np.uint8)
    lib().ora_tile_values(_p(values), N, K, _p(out))
    return out


def untile_values(tiled, N: int, K: int) -> np.ndarray:
    tiled = _c(tiled, np.uint8).ravel()
    out = np.empty((N, K // 2), dtype=np.uint8)
    lib().ora_untile_values(_p(tiled), N, K, _p(out))
    return out


def tile_meta(meta) -> np.ndarray:
    """Logical metadata [N, K/8] -> the ABI's tiled storage: contiguous
    128-row x 16-byte tiles."""
    meta = _c(meta, np.uint8)
    N, K = meta.shape[0], meta.shape[1] * 8
    out = np.empty(N * K // 8, dtype=np.uint8)
    lib().ora_tile_meta(_p(meta), N, K, _p(out))
    return out


def untile_meta(tiled, N: int, K: int) -> np.ndarray:
    tiled = _c(tiled, np.uint8).ravel()
    out = np.empty((N, K // 8), dtype=np.uint8)
    lib().ora_untile_meta(_p(tiled), N, K, _p(out))
    return out


def compress_abi(W_bits, gN: int = 1, gK: int = None):
    """compress() in the storage layout the C ABI produces and consumes."""
    values, meta, scales = compress(W_bits, gN, gK)
    return tile_values(values), tile_meta(meta), scales


# ------------------------------------------------------- activation quantize
def quantize_act(X, gK: int = None):
    """Per-token (gK = K) or 1 x gK activation quantization.
    Returns (xq uint8 [M,K], sx fp32 [K/gK, M])."""
    X = _c(X, np.float32)
    M, K = X.shape
    gK = K if gK is None else gK
    xq = np.empty((M, K), dtype=np.uint8)
    sx = np.empty((K // gK, M), dtype=np.float32)
    lib().ora_quantize_act(_p(X), M, K, K, gK, _p(xq), _p(sx))
    return xq, sx


# ---------------------------------------------------------------------- GEMM
def gemm(xq, sx, values, meta, sw, gM: int = 1, gN: int = 1, gK: int = None,
         X2=None, W2=None, acc_fp64: bool = False, bias=None) -> np.ndarray:
    """Group-wise scaled 2:4 sparse GEMM Y[M,N] = X.W^T (+ X2.W2^T) (+ bias), as float64.

    xq [M,K] e4m3; sx [K/gK, ceil(M/gM)]; values [N,K/2]; meta [N,K/8] logical;
    sw [K/gK, ceil(N/gN)]; X2 [M,r], W2 [N,r] bf16 bits or None; bias [N] bf16
    bits or None (the linear operation's bias, pytorch/ao PR #3258, added last).
    acc_fp64=False accumulates in fp32 (the reference the path is held to);
    True accumulates in double (used to bound the fp32 reference's own error).
    """
    xq = _c(xq, np.uint8)
    M, K = xq.shape
    gK = K if gK is None else gK
    values = _c(values, np.uint8)
    meta = _c(meta, np.uint8)
    N = values.shape[0]
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    assert sx.size == (K // gK) * ((M + gM - 1) // gM)
    assert sw.size == (K // gK) * ((N + gN - 1) // gN)
    r = 0
    if X2 is not None:
        X2 = _c(X2, np.uint16)
        W2 = _c(W2, np.uint16)
        r = X2.shape[1]
        assert X2.shape == (M, r) and W2.shape == (N, r)
    if bias is not None:
        bias = _c(bias, np.uint16)
        assert bias.shape == (N,)
    Y = np.empty((M, N), dtype=np.float64)
    lib().ora_gemm(_p(xq), _p(sx), M, K, K, gM, _p(values), _p(meta), _p(sw), N, gN, gK,
                   _p(X2), _p(W2), r, _p(bias), 1 if acc_fp64 else 0, _p(Y))
    return Y


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = _c(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, rounded to nearest, ties to even (finite
    inputs): add half an ulp of the kept 16 bits, plus the kept LSB for ties,
    then truncate."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def dequantize(values, meta, scales, gN: int = 1, gK: int = None) -> np.ndarray:
    """The dense dequantized weight as bf16 bits [N, K]: at the kept positions
    of every group of four, the e4m3 value times its block's weight scale
    (exact in double, then rounded to fp32, then to bf16); +0 at the pruned
    ones.  This is what the GEMM returns for an identity activation with unit
    activation scales (pytorch/ao PR #3258, dequantize by multiplying with an
    identity)."""
    codes = decompress(values, meta)
    N, K = codes.shape
    gK = K if gK is None else gK
    scales = _c(scales, np.float32)
    s = np.repeat(np.repeat(scales.astype(np.float64), gK, axis=0)[:K], gN, axis=1)[:, :N].T  # [N, K]
    prod = e4m3_decode(codes) * s          # exact: 4 x 24 significant bits
    return f32_to_bf16_bits(prod.astype(np.float32))


# --------------------------------------------------------------- int8 sibling
# The int8 x int8 2:4 sibling (pytorch/ao PR #3258, review: int8 x int8 and
# fp8 x fp8 are the 2:4 kernels; Int8SemiSparseTensor).  The pages define no
# int8 quantizer; sp24_oracle.c states the symmetric one taken here.
def int8_encode(x) -> int:
    """Nearest integer to x (fp32), ties to even, clamped to [-127, 127]."""
    return int(lib().ora_int8_from_f32(float(x)))


def compress_int8(W_bits):
    """Prune 2:4 and quantize to int8 with one scale per output channel.
    Returns (values int8 [N,K/2], meta uint8 [N,K/8] logical, scales fp32 [N])."""
    W_bits = _c(W_bits, np.uint16)
    N, K = W_bits.shape
    values = np.empty((N, K // 2), dtype=np.int8)
    meta = np.empty((N, K // 8), dtype=np.uint8)
    scales = np.empty(N, dtype=np.float32)
    lib().ora_compress_int8(_p(W_bits), N, K, K, _p(values), _p(meta), _p(scales))
    return values, meta, scales


def quantize_act_int8(X):
    """Per-token int8 activation quantization: (xq int8 [M,K], sx fp32 [M])."""
    X = _c(X, np.float32)
    M, K = X.shape
    xq = np.empty((M, K), dtype=np.int8)
    sx = np.empty(M, dtype=np.float32)
    lib().ora_quantize_act_int8(_p(X), M, K, K, _p(xq), _p(sx))
    return xq, sx


def gemm_int8(xq, sx, values, meta, sw, bias=None):
    """Y[M,N] (float64 of the fp32 result) and the exact int32 sums acc[M,N]."""
    xq = _c(xq, np.int8)
    M, K = xq.shape
    values = _c(values, np.int8)
    meta = _c(meta, np.uint8)
    N = values.shape[0]
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    assert sx.shape == (M,) and sw.shape == (N,) and K <= 131072
    if bias is not None:
        bias = _c(bias, np.uint16)
        assert bias.shape == (N,)
    Y = np.empty((M, N), dtype=np.float64)
    acc = np.empty((M, N), dtype=np.int32)
    lib().ora_gemm_int8(_p(xq), _p(sx), M, K, K, _p(values), _p(meta), _p(sw), N, _p(bias), _p(acc), _p(Y))
    return Y, acc
