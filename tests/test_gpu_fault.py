"""The give-up path of the bounded device waits, exercised without faulting
or hanging the GPU.

Every wait in the library's kernels gives up after a time limit, records a
bit in the device error word and unwinds (producers wait, bounded, for their
copies in flight; the MMA thread drains its MMAs; TMEM is freed), so that the
launch ends and sp24_last_device_error reports SP24_ERR_DEVICE_TIMEOUT.  This
test makes one such wait run out: a fault-test copy of the library, built
apart from libsp24.so with a 1 ms limit, issues nothing for the first
pipeline stage of each CTA of the one-CTA GEMM kernel, so that its MMA
thread waits for operands that never come.  No copy is in flight for the
withheld stage and no MMA runs on it.  The copy runs in a child process of
its own; the parent then checks that the library proper still computes the
oracle's result.
"""
import json
import subprocess
import sys

import pytest
import torch

import inputs
from gpu_util import assert_close, bf16_to_f64, dev

pytestmark = pytest.mark.gpu

SP24_ERR_DEVICE_TIMEOUT = 7

CHILD = r"""
import ctypes, json, sys
import torch
lib = ctypes.CDLL(sys.argv[1])
P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
lib.sp24_fp8_gemm.argtypes = [P, P, I64, I64, I64, I, P, P, P, I64, I, I, P, P, I64, P, P, I64, P, SZ, P]
lib.sp24_fp8_gemm.restype = I
lib.sp24_set_decomposition.argtypes = [I]
lib.sp24_set_decomposition.restype = I
lib.sp24_last_device_error.argtypes = [P]
lib.sp24_last_device_error.restype = I
ptr = lambda t: ctypes.c_void_p(t.data_ptr())
M, N, K = 64, 256, 512
xq = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
sx = torch.ones(M, dtype=torch.float32, device="cuda")
values = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
meta = torch.full((N, K // 8), 0x44, dtype=torch.uint8, device="cuda")  # valid nibbles: positions 0 and 1
sw = torch.ones(N, dtype=torch.float32, device="cuda")
y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
out = {"mode": lib.sp24_set_decomposition(1)}  # whole tiles: the one-CTA kernel, no split
out["launch"] = lib.sp24_fp8_gemm(ptr(xq), ptr(sx), M, K, K, 1, ptr(values), ptr(meta), ptr(sw), N, 1, K,
                                  None, None, 0, None, ptr(y), N, None, 0, s)
out["device"] = lib.sp24_last_device_error(s)
out["again"] = lib.sp24_last_device_error(s)  # the word was read and cleared
# the context still works after the launch gave up
out["context_ok"] = torch.arange(1000, device="cuda", dtype=torch.float32).sum().item() == 499500.0
print(json.dumps(out))
"""


def test_wait_timeout_is_reported_and_context_survives(ora, sp24):
    from semi_structured_sparse_gb300 import build as b
    fault_lib = b.build_fault_test()
    assert fault_lib != b.LIB
    r = subprocess.run([sys.executable, "-c", CHILD, fault_lib], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["mode"] == 0 and out["launch"] == 0
    assert out["device"] == SP24_ERR_DEVICE_TIMEOUT
    assert out["again"] == 0
    assert out["context_ok"]

    # the library proper, on the same shape and decomposition, in this process
    w = inputs.Workload("fault", 64, 256, 512, seed=41)
    X, W, _, _ = inputs.generate(w)
    xq, sx = ora.quantize_act(X.numpy(), w.gk)
    values, meta, sw = ora.compress(inputs.bf16_bits(W), w.gN, w.gk)
    tv, tm = ora.tile_values(values).reshape(w.N, -1), ora.tile_meta(meta).reshape(w.N, -1)
    with sp24.decomposition(sp24.DECOMP_DATA_PARALLEL):
        y = sp24.gemm(dev(xq), dev(sx), dev(tv), dev(tm), dev(sw), w.gM, w.gN, w.gk)
        torch.cuda.synchronize()
    sp24.last_device_error()
    assert_close(bf16_to_f64(y), ora.gemm(xq, sx, values, meta, sw, w.gM, w.gN, w.gk),
                 "library proper after the fault-test run")
