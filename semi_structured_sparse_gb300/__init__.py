"""semi_structured_sparse_gb300 -- Python binding of libsp24 (2:4 sparse FP8 GEMM on GB300).

Argument marshalling only: every step runs in the library's CUDA kernels.
torch supplies device memory and the current stream; the library itself never
allocates.  There is no CPU fallback: if the library is missing or the device
is not an sm_103 GPU, every call raises.

    values, meta, sw = compress(w_bf16, gN=1, gK=None)        # prune + e4m3 + pack
    xq, sx          = quantize_act(x_fp32, gK=None)            # per-token / 1x128 e4m3
    y               = gemm(xq, sx, values, meta, sw, gM=1, gN=1, gK=None, x2=None, w2=None)
"""
import contextlib
import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

SP24_STATUS = {
    0: "SP24_OK", 1: "SP24_ERR_INVALID_ARG", 2: "SP24_ERR_UNSUPPORTED", 3: "SP24_ERR_ALIGNMENT",
    4: "SP24_ERR_CUDA", 5: "SP24_ERR_ARCH", 6: "SP24_ERR_WORKSPACE", 7: "SP24_ERR_DEVICE_TIMEOUT",
}

# Every entry point the C header declares, with its ctypes signature.
_P, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "sp24_status_string": ([_I], ctypes.c_char_p),
    "sp24_meta_bytes": ([_I64, _I64], _SZ),
    "sp24_fp8_compress": ([_P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P], _I),
    "sp24_fp8_quantize_act": ([_P, _I64, _I64, _I64, _I, _P, _P, _P], _I),
    "sp24_fp8_quantize_act_bf16": ([_P, _I64, _I64, _I64, _I, _P, _P, _P], _I),
    "sp24_fp8_decompress": ([_P, _P, _P, _I64, _I64, _I, _I, _P, _I64, _P], _I),
    "sp24_fp8_gemm": ([_P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _I64, _I, _I, _P, _P, _I64, _P, _P, _I64,
                       _P, _SZ, _P], _I),
    "sp24_fp8_gemm_workspace_size": ([_I64, _I64, _I64, _I64], _SZ),
    "sp24_set_decomposition": ([_I], _I),
    "sp24_fp8_gemm_decomposition": ([_I64, _I64, _I64, _I64, _P], _I),
    "sp24_fp8_gemm_batched": ([_P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _I64, _I, _I, _P, _P, _I64, _I64,
                               _I64, _I64, _I64, _I64, _I64, _I64, _I64, _P, _SZ, _P], _I),
    "sp24_fp8_gemm_fixed_scratch": ([_P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _I64, _I, _I, _P, _P, _I64, _P, _P,
                                     _I64, _P], _I),
    "sp24_last_device_error": ([_P], _I),
    "sp24_int8_compress": ([_P, _I64, _I64, _I64, _P, _P, _P, _P], _I),
    "sp24_int8_quantize_act": ([_P, _I64, _I64, _I64, _P, _P, _P], _I),
    "sp24_int8_gemm": ([_P, _P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P, _I64, _P], _I),
}


class Sp24Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, SP24_STATUS.get(status, "status %d" % status)))


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libsp24.so (building it first if asked and it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libsp24.so is not built (run semi_structured_sparse_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        if status in (1, 2, 3):
            raise ValueError("%s: %s" % (where, SP24_STATUS.get(status, status)))
        raise Sp24Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev_tensor(t, dtype, name, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.stride(-1) != 1:
        raise ValueError("%s must have unit stride in its last dimension" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the operands on %s" % (name, t.device, device))
    return t


def _cdiv(a, b):
    return (a + b - 1) // b


def _scale_count(K, gK, rows, g):
    """Scales of a [rows, K] operand at granularity g x gK (0 if gK is invalid:
    the library then refuses the call itself)."""
    if not gK or K % gK != 0 or g <= 0:
        return 0
    return (K // gK) * _cdiv(rows, g)


def _at_least(t, n, name):
    """The kernels read or write n elements of t; the C ABI cannot see sizes."""
    if not t.is_contiguous() or t.numel() < n:
        raise ValueError("%s must be contiguous with at least %d elements (has %d)" % (name, n, t.numel()))


def _matrix(t, rows, cols, name):
    """A [rows, cols] matrix with unit column stride and row stride >= cols."""
    if t.dim() != 2 or tuple(t.shape) != (rows, cols) or t.stride(0) < cols:
        raise ValueError("%s must be [%d, %d], got %s" % (name, rows, cols, tuple(t.shape)))


def workspace_size(M: int, N: int, K: int, r: int = 0) -> int:
    """Device scratch bytes gemm() wants for this shape (0 = none)."""
    return int(load().sp24_fp8_gemm_workspace_size(M, N, K, r))


DECOMP_HEURISTIC, DECOMP_DATA_PARALLEL, DECOMP_STREAM_K, DECOMP_CLUSTER_SPLIT = 0, 1, 2, 3


def set_decomposition(mode: int) -> None:
    """How later GEMM calls deal out the tiles' K ranges: DECOMP_HEURISTIC
    (default), DECOMP_DATA_PARALLEL (whole tiles), DECOMP_STREAM_K or
    DECOMP_CLUSTER_SPLIT (process-wide; workspace_size() follows the mode)."""
    _check(load().sp24_set_decomposition(int(mode)), "sp24_set_decomposition")


@contextlib.contextmanager
def decomposition(mode: int):
    """Run a block of GEMM calls under one decomposition mode, then restore
    the heuristic."""
    set_decomposition(mode)
    try:
        yield
    finally:
        set_decomposition(DECOMP_HEURISTIC)


def decomposition_of(M: int, N: int, K: int, r: int = 0):
    """(mode, CTAs per tile) a per-tensor-K call of this shape would use now."""
    cs = ctypes.c_int(1)
    mode = int(load().sp24_fp8_gemm_decomposition(M, N, K, r, ctypes.addressof(cs)))
    if mode < 0:
        raise ValueError("invalid shape or no usable device")
    return mode, cs.value


def meta_bytes(N: int, K: int) -> int:
    return int(load().sp24_meta_bytes(N, K))


def compress(w: torch.Tensor, gN: int = 1, gK: int = None, out=None, stream=None):
    """Magnitude 2:4 prune + e4m3 + pack of a bf16 weight [N, K].

    Returns (values uint8 [N, K/2], meta uint8 [N, K/8], scales fp32 [K/gK, ceil(N/gN)]).
    values and meta hold the library's tiled storage (128 x 128 weight tiles,
    each contiguous; see include/sp24.h), which is what gemm() reads.
    ``out`` may supply those three tensors (no allocation then)."""
    lib = load()
    _dev_tensor(w, torch.bfloat16, "w")
    if w.dim() != 2:
        raise ValueError("w must be [N, K]")
    N, K = w.shape
    gK = K if gK is None else gK
    if out is None:
        values = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
        meta = torch.empty((N, K // 8), dtype=torch.uint8, device=w.device)
        scales = torch.empty((K // gK, (N + gN - 1) // gN), dtype=torch.float32, device=w.device)
    else:
        values, meta, scales = out
        _dev_tensor(values, torch.uint8, "values", w.device)
        _dev_tensor(meta, torch.uint8, "meta", w.device)
        _dev_tensor(scales, torch.float32, "scales", w.device)
        _at_least(values, N * (K // 2), "values")
        _at_least(meta, N * (K // 8), "meta")
        _at_least(scales, _scale_count(K, gK, N, gN), "scales")
    _check(lib.sp24_fp8_compress(_ptr(w), N, K, w.stride(0), gN, gK, _ptr(values), _ptr(meta), _ptr(scales),
                                 _stream(stream)), "sp24_fp8_compress")
    return values, meta, scales


def decompress(values, meta, scales, gN: int = 1, gK: int = None, out=None, stream=None):
    """The dense dequantized weight bf16 [N, K] from compress()'s output: at the
    kept positions bf16(scale * e4m3 value), 0 elsewhere."""
    lib = load()
    _dev_tensor(values, torch.uint8, "values")
    if values.dim() != 2:
        raise ValueError("values must be [N, K/2]")
    N, K = values.shape[0], values.shape[1] * 2
    gK = K if gK is None else gK
    _dev_tensor(meta, torch.uint8, "meta", values.device)
    _dev_tensor(scales, torch.float32, "scales", values.device)
    _at_least(values, N * (K // 2), "values")
    _at_least(meta, N * (K // 8), "meta")
    _at_least(scales, _scale_count(K, gK, N, gN), "scales")
    if out is None:
        W = torch.empty((N, K), dtype=torch.bfloat16, device=values.device)
    else:
        W = _dev_tensor(out, torch.bfloat16, "out", values.device)
        _matrix(W, N, K, "out")
    _check(lib.sp24_fp8_decompress(_ptr(values), _ptr(meta), _ptr(scales), N, K, gN, gK, _ptr(W), W.stride(0),
                                   _stream(stream)), "sp24_fp8_decompress")
    return W


def quantize_act(x: torch.Tensor, gK: int = None, out=None, stream=None):
    """Dynamic e4m3 quantization of fp32 or bf16 activations [M, K]: returns
    (xq uint8 [M, K], sx fp32 [K/gK, M])."""
    lib = load()
    bf16 = isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16
    _dev_tensor(x, torch.bfloat16 if bf16 else torch.float32, "x")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M, K = x.shape
    gK = K if gK is None else gK
    if out is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
        sx = torch.empty((K // gK, M), dtype=torch.float32, device=x.device)
    else:
        xq, sx = out
        _dev_tensor(xq, torch.uint8, "xq", x.device)
        _dev_tensor(sx, torch.float32, "sx", x.device)
        _at_least(xq, M * K, "xq")  # written densely, row stride K
        _at_least(sx, _scale_count(K, gK, M, 1), "sx")
    f, name = ((lib.sp24_fp8_quantize_act_bf16, "sp24_fp8_quantize_act_bf16") if bf16
               else (lib.sp24_fp8_quantize_act, "sp24_fp8_quantize_act"))
    _check(f(_ptr(x), M, K, x.stride(0), gK, _ptr(xq), _ptr(sx), _stream(stream)), name)
    return xq, sx


def gemm(xq, sx, values, meta, sw, gM: int = 1, gN: int = 1, gK: int = None, x2=None, w2=None,
         out=None, workspace=None, stream=None, bias=None):
    """Y[M, N] (bf16) = scaled 2:4 sparse e4m3 GEMM of xq [M, K] with the packed weight
    (values [N, K/2], meta [N, K/8]) plus x2 [M, r] . w2 [N, r]^T and a bf16 bias [N]
    when given.  `workspace` (uint8, at least workspace_size(M, N, K, r) bytes) must be
    zeroed before its first use and may then be reused by later calls of any shape on
    the same stream; without one, each call that needs scratch allocates a zeroed one."""
    lib = load()
    _dev_tensor(xq, torch.uint8, "xq")
    dev_ = xq.device
    _dev_tensor(values, torch.uint8, "values", dev_)
    if xq.dim() != 2 or values.dim() != 2:
        raise ValueError("xq must be [M, K] and values [N, K/2]")
    _dev_tensor(meta, torch.uint8, "meta", dev_)
    _dev_tensor(sx, torch.float32, "sx", dev_)
    _dev_tensor(sw, torch.float32, "sw", dev_)
    M, K = xq.shape
    N = values.shape[0]
    gK = K if gK is None else gK
    r = 0
    if x2 is not None:
        _dev_tensor(x2, torch.bfloat16, "x2", dev_)
        _dev_tensor(w2, torch.bfloat16, "w2", dev_)
        r = x2.shape[1]
        if not (x2.is_contiguous() and w2.is_contiguous()):
            raise ValueError("x2 and w2 must be contiguous")
        _matrix(x2, M, r, "x2")
        _matrix(w2, N, r, "w2")
    if not (sx.is_contiguous() and sw.is_contiguous() and values.is_contiguous() and meta.is_contiguous()):
        raise ValueError("scales, values and meta must be contiguous")
    _at_least(values, N * (K // 2), "values")
    _at_least(meta, N * (K // 8), "meta")
    _at_least(sx, _scale_count(K, gK, M, gM), "sx")
    _at_least(sw, _scale_count(K, gK, N, gN), "sw")
    if bias is not None:
        _dev_tensor(bias, torch.bfloat16, "bias", dev_)
        if not bias.is_contiguous() or bias.numel() != N:
            raise ValueError("bias must be a contiguous bf16 vector of N values")
    if out is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev_)
    else:
        y = _dev_tensor(out, torch.bfloat16, "out", dev_)
        _matrix(y, M, N, "out")
    ws_bytes = int(lib.sp24_fp8_gemm_workspace_size(M, N, K, r))
    if ws_bytes and workspace is None:
        workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev_)
    elif workspace is not None:
        _dev_tensor(workspace, torch.uint8, "workspace", dev_)
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
    _check(lib.sp24_fp8_gemm(_ptr(xq), _ptr(sx), M, K, xq.stride(0), gM, _ptr(values), _ptr(meta), _ptr(sw), N,
                             gN, gK, _ptr(x2), _ptr(w2), r, _ptr(bias), _ptr(y), y.stride(0), _ptr(workspace),
                             0 if workspace is None else workspace.numel() * workspace.element_size(),
                             _stream(stream)), "sp24_fp8_gemm")
    return y


def gemm_batched(xq, sx, values, meta, sw, gM: int = 1, gN: int = 1, gK: int = None, bias=None, out=None,
                 workspace=None, stream=None):
    """L independent problems of one shape: xq [L, M, K], sx [L, K/gK, ceil(M/gM)],
    values [L, N, K/2], meta [L, N, K/8], sw [L, K/gK, ceil(N/gN)], bias [L, N] or
    None -> Y [L, M, N] bf16, Y[l] = gemm(xq[l], ..., bias[l])."""
    lib = load()
    for t, dt, nm in ((xq, torch.uint8, "xq"), (values, torch.uint8, "values"), (meta, torch.uint8, "meta"),
                      (sx, torch.float32, "sx"), (sw, torch.float32, "sw")):
        _dev_tensor(t, dt, nm)
        if t.dim() != 3 or not t[0].is_contiguous():
            raise ValueError("%s must be [L, ...] with contiguous problems" % nm)
    L, M, K = xq.shape
    N = values.shape[1]
    gK = K if gK is None else gK
    dev_ = xq.device
    for t, nm in ((values, "values"), (meta, "meta"), (sx, "sx"), (sw, "sw")):
        if t.device != dev_ or t.shape[0] != L:
            raise ValueError("%s must hold the same L problems on %s" % (nm, dev_))
    _at_least(values[0], N * (K // 2), "values[l]")
    _at_least(meta[0], N * (K // 8), "meta[l]")
    _at_least(sx[0], _scale_count(K, gK, M, gM), "sx[l]")
    _at_least(sw[0], _scale_count(K, gK, N, gN), "sw[l]")
    if bias is not None:
        _dev_tensor(bias, torch.bfloat16, "bias", dev_)
        if bias.shape != (L, N):
            raise ValueError("bias must be [L, N]")
    if out is None:
        y = torch.empty((L, M, N), dtype=torch.bfloat16, device=dev_)
    else:
        y = _dev_tensor(out, torch.bfloat16, "out", dev_)
        if y.dim() != 3 or tuple(y.shape) != (L, M, N) or y.stride(1) < N:
            raise ValueError("out must be [L, M, N]")
    ws_bytes = L * int(lib.sp24_fp8_gemm_workspace_size(M, N, K, 0))
    if ws_bytes and workspace is None:
        workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev_)
    elif workspace is not None:
        _dev_tensor(workspace, torch.uint8, "workspace", dev_)
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
    _check(lib.sp24_fp8_gemm_batched(
        _ptr(xq), _ptr(sx), M, K, xq.stride(1), gM, _ptr(values), _ptr(meta), _ptr(sw), N, gN, gK, _ptr(bias),
        _ptr(y), y.stride(1), L, xq.stride(0), sx.stride(0), values.stride(0), meta.stride(0), sw.stride(0),
        0 if bias is None else bias.stride(0), y.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream)),
        "sp24_fp8_gemm_batched")
    return y


# --------------------------------------------------------------- int8 sibling
def compress_int8(w: torch.Tensor, out=None, stream=None):
    """Magnitude 2:4 prune + int8 (one scale per output channel) + pack of a bf16
    weight [N, K]: (values int8 [N, K/2], meta uint8 [N, K/8], scales fp32 [N]),
    values and meta in the tiled storage gemm_int8() reads."""
    lib = load()
    _dev_tensor(w, torch.bfloat16, "w")
    if w.dim() != 2:
        raise ValueError("w must be [N, K]")
    N, K = w.shape
    if out is None:
        values = torch.empty((N, K // 2), dtype=torch.int8, device=w.device)
        meta = torch.empty((N, K // 8), dtype=torch.uint8, device=w.device)
        scales = torch.empty(N, dtype=torch.float32, device=w.device)
    else:
        values, meta, scales = out
        _dev_tensor(values, torch.int8, "values", w.device)
        _dev_tensor(meta, torch.uint8, "meta", w.device)
        _dev_tensor(scales, torch.float32, "scales", w.device)
        _at_least(values, N * (K // 2), "values")
        _at_least(meta, N * (K // 8), "meta")
        _at_least(scales, N, "scales")
    _check(lib.sp24_int8_compress(_ptr(w), N, K, w.stride(0), _ptr(values), _ptr(meta), _ptr(scales),
                                  _stream(stream)), "sp24_int8_compress")
    return values, meta, scales


def quantize_act_int8(x: torch.Tensor, out=None, stream=None):
    """Per-token int8 quantization of fp32 activations [M, K]: (xq int8 [M, K], sx fp32 [M])."""
    lib = load()
    _dev_tensor(x, torch.float32, "x")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M, K = x.shape
    if out is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
        sx = torch.empty(M, dtype=torch.float32, device=x.device)
    else:
        xq, sx = out
        _dev_tensor(xq, torch.int8, "xq", x.device)
        _dev_tensor(sx, torch.float32, "sx", x.device)
        _matrix(xq, M, K, "xq")
        if not xq.is_contiguous():
            raise ValueError("xq must be contiguous")
        _at_least(sx, M, "sx")
    _check(lib.sp24_int8_quantize_act(_ptr(x), M, K, x.stride(0), _ptr(xq), _ptr(sx), _stream(stream)),
           "sp24_int8_quantize_act")
    return xq, sx


def gemm_int8(xq, sx, values, meta, sw, bias=None, out=None, stream=None):
    """Y[M, N] bf16 = bf16((sx[m] sw[n]) * float(sum of the kept xq[m, k] wq[n, k]) + bias[n])
    for int8 activations xq [M, K] and compress_int8()'s packed weight."""
    lib = load()
    _dev_tensor(xq, torch.int8, "xq")
    dev_ = xq.device
    _dev_tensor(values, torch.int8, "values", dev_)
    if xq.dim() != 2 or values.dim() != 2:
        raise ValueError("xq must be [M, K] and values [N, K/2]")
    _dev_tensor(meta, torch.uint8, "meta", dev_)
    _dev_tensor(sx, torch.float32, "sx", dev_)
    _dev_tensor(sw, torch.float32, "sw", dev_)
    M, K = xq.shape
    N = values.shape[0]
    if not (sx.is_contiguous() and sw.is_contiguous() and values.is_contiguous() and meta.is_contiguous()):
        raise ValueError("scales, values and meta must be contiguous")
    _at_least(values, N * (K // 2), "values")
    _at_least(meta, N * (K // 8), "meta")
    _at_least(sx, M, "sx")
    _at_least(sw, N, "sw")
    if bias is not None:
        _dev_tensor(bias, torch.bfloat16, "bias", dev_)
        if not bias.is_contiguous() or bias.numel() != N:
            raise ValueError("bias must be a contiguous bf16 vector of N values")
    if out is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev_)
    else:
        y = _dev_tensor(out, torch.bfloat16, "out", dev_)
        _matrix(y, M, N, "out")
    _check(lib.sp24_int8_gemm(_ptr(xq), _ptr(sx), M, K, xq.stride(0), _ptr(values), _ptr(meta), _ptr(sw), N,
                              _ptr(bias), _ptr(y), y.stride(0), _stream(stream)), "sp24_int8_gemm")
    return y


def last_device_error(stream=None):
    """Synchronise and raise if any library kernel gave up on a bounded wait."""
    _check(load().sp24_last_device_error(_stream(stream)), "device")
