"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every symbol include/sp24.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sp24.h")


@pytest.fixture(scope="module")
def lib():
    import semi_structured_sparse_gb300 as s
    return s.load()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"SP24_API\s+[\w\s\*]*?\b(sp24_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("sp24_fp8_compress", "sp24_fp8_gemm", "sp24_fp8_quantize_act",
                     "sp24_fp8_gemm_workspace_size", "sp24_meta_bytes", "sp24_status_string",
                     "sp24_last_device_error"):
        assert required in names


def test_exports_every_declared_symbol(lib):
    import semi_structured_sparse_gb300 as s
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in s.SIGNATURES, name


def test_status_strings(lib):
    for code in range(8):
        assert lib.sp24_status_string(code).startswith(b"SP24_")
    assert lib.sp24_status_string(99) == b"SP24_ERR_UNKNOWN"


def test_meta_bytes(lib):
    assert lib.sp24_meta_bytes(4096, 4096) == 4096 * 512
    assert lib.sp24_meta_bytes(1, 8) == 1
    assert lib.sp24_meta_bytes(0, 128) == 0
    assert lib.sp24_meta_bytes(4, 12) == 0


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x10008)  # 8-byte aligned only


def test_compress_argument_errors(lib):
    f = lib.sp24_fp8_compress
    ok = dict(W=FAKE, N=256, K=512, ldw=512, gN=1, gK=512, v=FAKE, m=FAKE, s=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["W"], a["N"], a["K"], a["ldw"], a["gN"], a["gK"], a["v"], a["m"], a["s"], None)

    assert call(W=None) == 1
    assert call(v=None) == 1
    assert call(N=0) == 1
    assert call(K=100) == 1          # not a multiple of 128
    assert call(ldw=256) == 1        # stride shorter than a row
    assert call(gN=2) == 2
    assert call(gN=128, gK=512) == 2
    assert call(gN=128, gK=128, N=200) == 1
    assert call(N=100) == 1          # tiled storage: whole 128-row bands
    assert call(W=FAKE_ODD) == 3
    assert call(ldw=516) == 3        # row stride not 16-byte aligned


def test_gemm_argument_errors(lib):
    f = lib.sp24_fp8_gemm
    ok = dict(X=FAKE, sx=FAKE, M=64, K=512, ldx=512, gM=1, v=FAKE, m=FAKE, sw=FAKE, N=256, gN=1, gK=512,
              X2=None, W2=None, r=0, bias=None, Y=FAKE, ldy=256)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["X"], a["sx"], a["M"], a["K"], a["ldx"], a["gM"], a["v"], a["m"], a["sw"], a["N"], a["gN"],
                 a["gK"], a["X2"], a["W2"], a["r"], a["bias"], a["Y"], a["ldy"], None, 0, None)

    assert call(X=None) == 1
    assert call(Y=None) == 1
    assert call(M=0) == 1
    assert call(N=200) == 1           # N must be a multiple of 128
    assert call(K=200) == 1
    assert call(ldx=256) == 1
    assert call(ldy=128) == 1
    assert call(gM=2) == 2
    assert call(gK=256) == 2
    assert call(r=64) == 1            # side rank without operands
    assert call(r=24, X2=FAKE, W2=FAKE) == 2
    assert call(r=128, X2=FAKE, W2=FAKE) == 2
    assert call(X=FAKE_ODD) == 3
    assert call(ldx=520) == 3
    assert call(ldy=260) == 3        # output rows must stay 16-byte aligned
    assert call(bias=ctypes.c_void_p(0x10001)) == 3  # bf16 bias: 2-byte aligned


def test_quantize_argument_errors(lib):
    f = lib.sp24_fp8_quantize_act
    assert f(None, 4, 128, 128, 128, FAKE, FAKE, None) == 1
    assert f(FAKE, 4, 100, 128, 128, FAKE, FAKE, None) == 1
    assert f(FAKE, 4, 256, 256, 64, FAKE, FAKE, None) == 2
    assert f(FAKE_ODD, 4, 256, 256, 128, FAKE, FAKE, None) == 3
    g = lib.sp24_fp8_quantize_act_bf16
    assert g(None, 4, 128, 128, 128, FAKE, FAKE, None) == 1
    assert g(FAKE, 4, 256, 200, 128, FAKE, FAKE, None) == 1   # ldx < K
    assert g(FAKE, 4, 256, 256, 64, FAKE, FAKE, None) == 2
    assert g(FAKE, 4, 256, 260, 128, FAKE, FAKE, None) == 3   # bf16 rows: 16-byte multiples
    assert g(FAKE_ODD, 4, 256, 256, 128, FAKE, FAKE, None) == 3


def test_decompress_argument_errors(lib):
    f = lib.sp24_fp8_decompress
    assert f(None, FAKE, FAKE, 128, 256, 1, 256, FAKE, 256, None) == 1
    assert f(FAKE, FAKE, FAKE, 100, 256, 1, 256, FAKE, 256, None) == 1   # whole 128-row bands
    assert f(FAKE, FAKE, FAKE, 128, 200, 1, 200, FAKE, 256, None) == 1
    assert f(FAKE, FAKE, FAKE, 128, 256, 1, 256, FAKE, 128, None) == 1   # ldw < K
    assert f(FAKE, FAKE, FAKE, 128, 256, 128, 256, FAKE, 256, None) == 2  # 128 x K blocks: not a compress output
    assert f(FAKE, FAKE, FAKE, 128, 256, 1, 256, FAKE, 260, None) == 3   # bf16 rows: 16-byte multiples
    assert f(FAKE, FAKE, FAKE, 128, 256, 1, 256, FAKE_ODD, 256, None) == 3


def test_gemm_batched_argument_errors(lib):
    f = lib.sp24_fp8_gemm_batched

    def call(L=2, sxq=64 * 512, sv=256 * 256, sm=256 * 64, ssx=64, ssw=256, sb=0, sy=64 * 256, bias=None):
        return f(FAKE, FAKE, 64, 512, 512, 1, FAKE, FAKE, FAKE, 256, 1, 512, bias, FAKE, 256, L,
                 sxq, ssx, sv, sm, ssw, sb, sy, None, 0, None)

    assert call(L=0) == 1
    assert call(sxq=64 * 512 - 16) == 1   # problems overlap
    assert call(sv=100) == 1
    assert call(bias=FAKE, sb=100) == 1   # bias rows overlap
    assert call(sxq=64 * 512 + 8) == 3    # not a 16-byte multiple
    assert call(sy=64 * 256 + 4) == 3


def test_workspace_size(lib):
    assert lib.sp24_fp8_gemm_workspace_size(2048, 4096, 4096, 0) >= 0


def test_set_decomposition_modes(lib):
    """The three modes are accepted, anything else refused; the heuristic is
    left in force."""
    try:
        for mode in (1, 2, 3, 0):
            assert lib.sp24_set_decomposition(mode) == 0
        for bad in (-1, 4, 100):
            assert lib.sp24_set_decomposition(bad) == 1  # SP24_ERR_INVALID_ARG
    finally:
        lib.sp24_set_decomposition(0)


def test_product_path_has_no_cpu_fallback():
    """The binding never routes through the oracle or a CPU implementation."""
    pkg = os.path.join(ROOT, "semi_structured_sparse_gb300", "__init__.py")
    txt = open(pkg).read()
    assert "import oracle" not in txt and "from oracle" not in txt
    assert "import numpy" not in txt


def test_binding_size_checks():
    """The binding checks what the C ABI cannot see: buffer sizes, shapes and
    strides of the tensors the kernels read and write."""
    import torch
    import semi_structured_sparse_gb300 as s
    assert s._scale_count(4096, 4096, 2048, 1) == 2048          # per token
    assert s._scale_count(4096, 128, 3000, 1) == 32 * 3000      # 1 x 128
    assert s._scale_count(4096, 128, 300, 128) == 32 * 3        # 128 x 128, ragged
    assert s._scale_count(4096, 100, 16, 1) == 0                # invalid gK: the library refuses it
    s._at_least(torch.zeros(10), 10, "t")
    with pytest.raises(ValueError):
        s._at_least(torch.zeros(9), 10, "t")
    with pytest.raises(ValueError):
        s._at_least(torch.zeros(4, 6)[:, :3], 12, "t")             # not contiguous
    s._matrix(torch.zeros(4, 8)[:, :6], 4, 6, "m")                # a row stride above the width is fine
    with pytest.raises(ValueError):
        s._matrix(torch.zeros(4, 6), 4, 8, "m")
    with pytest.raises(ValueError):
        s._matrix(torch.zeros(24), 4, 6, "m")
    with pytest.raises(ValueError):
        s._dev_tensor(torch.zeros(4), torch.float32, "t")          # host tensors are refused


def test_fault_switches_stay_out_of_the_library():
    """The give-up-path test library is built apart, with its own switches;
    the library proper is compiled without them."""
    from semi_structured_sparse_gb300 import build as b
    assert b.FAULT_LIB != b.LIB and os.path.dirname(b.FAULT_LIB) != os.path.dirname(b.LIB)
    assert not any("SP24_FAULT" in f or "SP24_WAIT_TIMEOUT_NS" in f for f in b.FLAGS)
    assert any("SP24_FAULT_WITHHOLD_FIRST_STAGE" in f for f in b.FAULT_FLAGS)


def test_int8_argument_errors(lib):
    """The int8 sibling's entry points refuse bad arguments before any launch."""
    P = ctypes.c_void_p
    one = P(16)
    INVALID, UNSUPPORTED = 1, 2  # SP24_ERR_INVALID_ARG, SP24_ERR_UNSUPPORTED
    # compress: N not a multiple of 128, K not a multiple of 128, null pointers
    assert lib.sp24_int8_compress(one, 100, 256, 256, one, one, one, None) == INVALID
    assert lib.sp24_int8_compress(one, 128, 200, 200, one, one, one, None) == INVALID
    assert lib.sp24_int8_compress(None, 128, 256, 256, one, one, one, None) == INVALID
    # quantize: K not a multiple of 128, ldx < K
    assert lib.sp24_int8_quantize_act(one, 4, 100, 100, one, one, None) == INVALID
    assert lib.sp24_int8_quantize_act(one, 4, 256, 128, one, one, None) == INVALID
    # gemm: K above the exact-int32 bound, N not a multiple of 128, ldy < N
    assert lib.sp24_int8_gemm(one, one, 4, 131200, 131200, one, one, one, 128, None, one, 128, None) == UNSUPPORTED
    assert lib.sp24_int8_gemm(one, one, 4, 256, 256, one, one, one, 100, None, one, 128, None) == INVALID
    assert lib.sp24_int8_gemm(one, one, 4, 256, 256, one, one, one, 128, None, one, 64, None) == INVALID
