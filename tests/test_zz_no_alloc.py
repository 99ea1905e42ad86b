"""sp24_fp8_gemm_fixed_scratch: the GEMM for callers that may not allocate.

Such callers (serving loops with every buffer planned at start-up, code hosted
in a framework whose allocator this library cannot reach) get the stream-K
scratch from a fixed array inside the library instead of a workspace they pass
in.  This file checks, through the C ABI, that two calls in a row give the same
result as sp24_fp8_gemm with a caller workspace (within the suite's tolerance),
and that a shape needing more scratch than the fixed array is refused.

It sits in its own file, collected last, so that a run which stops at the
first failure has already run every other test; it also passes on its own in
a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import inputs
from gpu_util import assert_close, bf16_to_f64, dev

pytestmark = pytest.mark.gpu

FIXED_SCRATCH_BYTES = 8 << 20   # the array size the header documents
SP24_ERR_WORKSPACE = 6


def _operands(ora, w):
    X, W, _, _ = inputs.generate(w)
    xq, sx = ora.quantize_act(X.numpy())
    values, meta, sw = ora.compress(inputs.bf16_bits(W))
    N = values.shape[0]
    tv = ora.tile_values(values).reshape(N, -1)
    tm = ora.tile_meta(meta).reshape(N, -1)
    return [dev(a) for a in (xq, sx, tv, tm, sw)], (xq, sx, values, meta, sw)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _gemm_with_workspace(lib, d, M, N, K, ws):
    xq, sx, tv, tm, sw = d
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.sp24_fp8_gemm(_p(xq), _p(sx), M, K, K, 1, _p(tv), _p(tm), _p(sw), N, 1, K, None, None, 0, None,
                           _p(y), N, _p(ws), ws.numel(), _stream())
    return st, y


def _gemm_fixed_scratch(lib, d, M, N, K):
    xq, sx, tv, tm, sw = d
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.sp24_fp8_gemm_fixed_scratch(_p(xq), _p(sx), M, K, K, 1, _p(tv), _p(tm), _p(sw), N, 1, K, None, None,
                                         0, None, _p(y), N, _stream())
    return st, y


@pytest.fixture
def streamk(sp24):
    """Stream-K forced, so that the small shapes below need scratch."""
    sp24.set_decomposition(sp24.DECOMP_STREAM_K)
    yield
    sp24.set_decomposition(sp24.DECOMP_HEURISTIC)


def test_fixed_scratch_matches_workspace_entry_point(ora, sp24, streamk):
    lib = sp24.load()
    M, N, K = 16, 5120, 4096          # few tiles: the GEMM splits K and needs scratch
    need = lib.sp24_fp8_gemm_workspace_size(M, N, K, 0)
    assert 0 < need <= FIXED_SCRATCH_BYTES
    d, host = _operands(ora, inputs.Workload("na", M, N, K, seed=31))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    st, y_ref = _gemm_with_workspace(lib, d, M, N, K, ws)
    assert st == 0
    ref = bf16_to_f64(y_ref)
    for call in range(2):             # the array keeps the previous call's contents
        st, y = _gemm_fixed_scratch(lib, d, M, N, K)
        assert st == 0, "call %d returned status %d" % (call, st)
        torch.cuda.synchronize()
        sp24.last_device_error()
        assert_close(bf16_to_f64(y), ref, "fixed-scratch call %d vs workspace entry point" % call)
    # and both agree with the oracle
    assert_close(ref, ora.gemm(*host), "workspace entry point vs oracle")


def test_fixed_scratch_refuses_oversized_shapes(ora, sp24, streamk):
    lib = sp24.load()
    M, N, K = 64, 4096, 4096          # the largest stream-K partials (64-token tiles)
    need = lib.sp24_fp8_gemm_workspace_size(M, N, K, 0)
    d, _ = _operands(ora, inputs.Workload("na2", M, N, K, seed=32))
    st, y = _gemm_fixed_scratch(lib, d, M, N, K)
    if need > FIXED_SCRATCH_BYTES:
        assert st == SP24_ERR_WORKSPACE
    else:                              # another SM count may split less: then it must just work
        assert st == 0
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
        st2, y_ref = _gemm_with_workspace(lib, d, M, N, K, ws)
        assert st2 == 0
        torch.cuda.synchronize()
        assert_close(bf16_to_f64(y), bf16_to_f64(y_ref), "fixed-scratch vs workspace entry point")
