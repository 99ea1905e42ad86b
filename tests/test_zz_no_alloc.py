"""sp24_fp8_gemm_fixed_scratch: the GEMM for callers that may not allocate.

Such callers (serving loops with every buffer planned at start-up, code hosted
in a framework whose allocator this library cannot reach) get the stream-K
scratch from a fixed array inside the library instead of a workspace they pass
in.  This file checks, through the C ABI, that two calls in a row give the same
result as sp24_fp8_gemm with a caller workspace (within the suite's tolerance),
that the shape with the largest scratch need fits the array, and that calls
allocate no device memory.

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


def test_fixed_scratch_largest_streamk_shape(ora, sp24, streamk):
    """The shape with the largest stream-K scratch (64-token tiles, one partial
    per SM) fits the fixed array on this part, and runs.  The library refuses
    a shape that needs more than the array holds (SP24_ERR_WORKSPACE); a
    compile-time bound in the library keeps every shape within it on parts
    with up to 240 SMs, so that refusal only guards larger parts."""
    lib = sp24.load()
    M, N, K = 64, 4096, 4096
    need = lib.sp24_fp8_gemm_workspace_size(M, N, K, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms <= 240 and 0 < need <= FIXED_SCRATCH_BYTES
    d, host = _operands(ora, inputs.Workload("na2", M, N, K, seed=32))
    st, y = _gemm_fixed_scratch(lib, d, M, N, K)
    assert st == 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    st2, y_ref = _gemm_with_workspace(lib, d, M, N, K, ws)
    assert st2 == 0
    torch.cuda.synchronize()
    sp24.last_device_error()
    assert_close(bf16_to_f64(y), bf16_to_f64(y_ref), "fixed-scratch vs workspace entry point")
    assert_close(bf16_to_f64(y), ora.gemm(*host), "fixed-scratch vs oracle")


def test_fixed_scratch_allocates_nothing(ora, sp24, streamk):
    """After a first call (which may load the library's device image), further
    calls change neither the memory torch has allocated on the device nor the
    device's free memory: the scratch is the library's own resident array."""
    lib = sp24.load()
    M, N, K = 32, 5120, 4096
    assert lib.sp24_fp8_gemm_workspace_size(M, N, K, 0) > 0   # the call does use scratch
    d, _ = _operands(ora, inputs.Workload("na3", M, N, K, seed=33))
    xq, sx, tv, tm, sw = d
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def call():
        return lib.sp24_fp8_gemm_fixed_scratch(_p(xq), _p(sx), M, K, K, 1, _p(tv), _p(tm), _p(sw), N, 1, K, None,
                                               None, 0, None, _p(y), N, _stream())

    assert call() == 0
    torch.cuda.synchronize()
    allocated = torch.cuda.memory_allocated()
    free, _ = torch.cuda.mem_get_info()
    for _ in range(4):
        assert call() == 0
    torch.cuda.synchronize()
    sp24.last_device_error()
    assert torch.cuda.memory_allocated() == allocated
    assert torch.cuda.mem_get_info()[0] == free
