"""GPU parity of the int8 x int8 2:4 sibling against the CPU oracle, through
the C ABI: compression and activation quantization bit-exact, and the GEMM's
bf16 output bit-exact too (its integer sums are exact and its epilogue rounds
the same fp32 steps as the oracle, then to bf16)."""
import numpy as np
import pytest
import torch

import inputs
from gpu_util import dev, host_bits

pytestmark = pytest.mark.gpu


def _weights(N, K, seed):
    _, W, _, _ = inputs.generate(inputs.Workload("i8", 1, N, K, seed=seed))
    return W


def _compress_both(ora, sp24, W):
    ov, om, os_ = ora.compress_int8(inputs.bf16_bits(W))
    gv, gm, gs = sp24.compress_int8(W.cuda())
    torch.cuda.synchronize()
    sp24.last_device_error()
    N, K = W.shape
    tv = ora.tile_values(ov.view(np.uint8)).reshape(N, -1)
    tm = ora.tile_meta(om).reshape(N, -1)
    return (tv, tm, os_), (gv.cpu().numpy().view(np.uint8), gm.cpu().numpy(), gs.cpu().numpy())


@pytest.mark.parametrize("N,K", [(128, 256), (256, 2048), (384, 4096), (128, 2176), (256, 8192), (128, 12288),
                                 (128, 20480)])
def test_int8_compress_bit_exact(ora, sp24, N, K):
    """Rows held by a persistent warp pair (K <= 4096), by 4 or 8 warps, longer
    rows streamed twice, and a ragged last chunk (K % 256 == 128)."""
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, _weights(N, K, N + K))
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(gm, om)
    assert np.array_equal(gv, ov)


def test_int8_compress_edge_values(ora, sp24):
    """Ties, signed zeros, all-zero rows, subnormal bf16, huge values."""
    N, K = 128, 512
    rng = np.random.default_rng(13)
    vals = np.array([0.0, -0.0, 1.0, -1.0, 2.0, 1e-38, -3e-39, 3e38, -1.5, 0.5, 127.0], dtype=np.float32)
    W = torch.from_numpy(rng.choice(vals, size=(N, K)).astype(np.float32)).to(torch.bfloat16)
    W[3] = 0.0
    W[4] = -0.0
    W[5, :] = 7.0
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(gm, om)
    assert np.array_equal(gv, ov)


@pytest.mark.parametrize("M,K", [(1, 128), (7, 4096), (300, 1024)])
def test_int8_quantize_act_bit_exact(ora, sp24, M, K):
    rng = np.random.default_rng(M + K)
    X = rng.normal(size=(M, K)).astype(np.float32)
    if M > 3:
        X[2] = 0.0
        X[3, :5] = [0.5, -0.5, 1.5, 2.5, -2.5]
    oq, osx = ora.quantize_act_int8(X)
    gq, gsx = sp24.quantize_act_int8(torch.from_numpy(X).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(gsx.cpu().numpy().view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(gq.cpu().numpy(), oq)


def _gemm_case(ora, sp24, M, N, K, seed, with_bias):
    w = inputs.Workload("i8g", M, N, K, seed=seed)
    X, W, _, _ = inputs.generate(w)
    values, meta, sw = ora.compress_int8(inputs.bf16_bits(W))
    xq, sx = ora.quantize_act_int8(X.numpy())
    bias = None
    if with_bias:
        rng = np.random.default_rng(seed)
        bias = inputs.bf16_bits(torch.from_numpy(rng.normal(size=N).astype(np.float32)).to(torch.bfloat16))
    Y, acc = ora.gemm_int8(xq, sx, values, meta, sw, bias=bias)
    tv = ora.tile_values(values.view(np.uint8)).reshape(N, -1)
    tm = ora.tile_meta(meta).reshape(N, -1)
    y = sp24.gemm_int8(dev(xq), dev(sx), dev(tv.view(np.int8)), dev(tm), dev(sw),
                       bias=None if bias is None else dev(bias))
    torch.cuda.synchronize()
    sp24.last_device_error()
    want = ora.f32_to_bf16_bits(Y.astype(np.float32))
    return host_bits(y), want, acc


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (7, 256, 512), (64, 128, 4096), (65, 384, 1024), (100, 256, 2176),
                                   (301, 640, 768)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_int8_gemm_bit_exact(ora, sp24, M, N, K, with_bias):
    """Token tails inside a 64-token tile and past a 32-token warp half, a
    single 128-wide K block, K blocks not a multiple of the 64-wide slices'
    pairs, several weight-row tiles."""
    got, want, _ = _gemm_case(ora, sp24, M, N, K, M * 7 + N + K, with_bias)
    assert np.array_equal(got, want)


def test_int8_gemm_full_size(ora, sp24):
    """The Llama-style linear's shape (M 2048, N 4096, K 4096), every element."""
    got, want, acc = _gemm_case(ora, sp24, 2048, 4096, 4096, 4, True)
    assert np.abs(acc).max() > 1000  # the comparison is not vacuous
    assert np.array_equal(got, want)


def test_int8_compress_then_gemm_on_device(ora, sp24):
    """compress_int8 and quantize_act_int8 on the device feed gemm_int8 directly."""
    w = inputs.Workload("i8d", 130, 512, 1024, seed=23)
    X, W, _, _ = inputs.generate(w)
    values, meta, sw = sp24.compress_int8(W.cuda())
    xq, sx = sp24.quantize_act_int8(X.cuda())
    y = sp24.gemm_int8(xq, sx, values, meta, sw)
    torch.cuda.synchronize()
    sp24.last_device_error()
    ov, om, osw = ora.compress_int8(inputs.bf16_bits(W))
    oq, osx = ora.quantize_act_int8(X.numpy())
    Y, _ = ora.gemm_int8(oq, osx, ov, om, osw)
    assert np.array_equal(host_bits(y), ora.f32_to_bf16_bits(Y.astype(np.float32)))
