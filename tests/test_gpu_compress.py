"""GPU parity of the weight compression and the activation quantization:
bit-exact against the CPU oracle (values, metadata and scales), through the
C ABI, on every workload's weight at full size."""
import numpy as np
import pytest
import torch

import inputs
from gpu_util import dev, host_bits

pytestmark = pytest.mark.gpu


def _compress_both(ora, sp24, Wt, gN, gK):
    Wb = inputs.bf16_bits(Wt)
    ov, om, os_ = ora.compress_abi(Wb, gN, gK)
    gv, gm, gs = sp24.compress(dev(Wb), gN, gK)
    torch.cuda.synchronize()
    sp24.last_device_error()
    return (ov, om, os_), (host_bits(gv).ravel(), host_bits(gm).ravel(), host_bits(gs))


@pytest.mark.parametrize("name", ["tiny", "llama", "groupwise", "decode"])
def test_compress_bit_exact_full_size(ora, sp24, name):
    w = inputs.WORKLOADS[name]
    _, W, _, _ = inputs.generate(inputs.with_shape(w, M=1))
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W, w.gN, w.gk)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), "scales"
    assert np.array_equal(gm, om), "metadata"
    assert np.array_equal(gv, ov), "values"


@pytest.mark.parametrize("gN,gK", [(1, None), (1, 128), (128, 128)])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 4352), (128, 640)])
def test_compress_ragged_shapes(ora, sp24, N, K, gN, gK):
    _, W, _, _ = inputs.generate(inputs.Workload("t", 1, N, K, seed=N + K))
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W, gN, K if gK is None else gK)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(gm, om)
    assert np.array_equal(gv, ov)


@pytest.mark.parametrize("N,K", [(256, 2048), (128, 2176), (384, 3072), (128, 5120), (256, 8192), (128, 12288),
                                 (128, 16384), (128, 16512), (128, 20480)])
def test_compress_row_lengths(ora, sp24, N, K):
    """Per-channel compression across row lengths: rows held in registers
    whole by a persistent warp pair that prefetches its next row (K <= 4096),
    by 4 warps (K <= 8192) or 8 warps (K <= 16384), rows longer than that
    whose amax pass streams past the held chunks, and ragged final chunks
    (K % 256 == 128)."""
    _, W, _, _ = inputs.generate(inputs.Workload("rl", 1, N, K, seed=N ^ K))
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W, 1, K)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(gm, om)
    assert np.array_equal(gv, ov)


def test_compress_many_rows_per_cta(ora, sp24):
    """Many short rows: each warp pair of the persistent kernel walks 13 or 14
    of them (both row buffers, an odd count ending early), most chunks idle."""
    _, W, _, _ = inputs.generate(inputs.Workload("mr", 1, 16384, 256, seed=3))
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W, 1, 256)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(gm, om)
    assert np.array_equal(gv, ov)


def test_compress_edge_values(ora, sp24):
    """Ties, signed zeros, an all-zero row, subnormal bf16 and huge values."""
    N, K = 128, 256
    rng = np.random.default_rng(5)
    vals = np.array([0.0, -0.0, 1.0, -1.0, 2.0, 1e-38, -3e-39, 3e38, -1.5, 0.5], dtype=np.float32)
    W = torch.from_numpy(rng.choice(vals, size=(N, K)).astype(np.float32)).to(torch.bfloat16)
    W[3] = 0.0          # all-zero row: scale 1, codes 0
    W[4] = -0.0
    W[5, :] = 7.0       # all ties
    (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W, 1, K)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(gm, om)
    assert np.array_equal(gv, ov)
    assert gs[0, 3] == 1.0


def test_compress_all_zero_weight(ora, sp24):
    W = torch.zeros((256, 512), dtype=torch.bfloat16)
    for gN, gK in [(1, 512), (1, 128), (128, 128)]:
        (ov, om, os_), (gv, gm, gs) = _compress_both(ora, sp24, W, gN, gK)
        assert (gs == 1.0).all() and (gv == 0).all() and (gm == 0x44).all()


def test_compress_strided_input(ora, sp24):
    """Row stride larger than K (a view into a wider weight)."""
    _, Wbig, _, _ = inputs.generate(inputs.Workload("t", 1, 256, 1024, seed=12))
    W = Wbig[:, :512]
    Wd = dev(inputs.bf16_bits(Wbig))[:, :512]
    gv, gm, gs = sp24.compress(Wd, 1, 512)
    ov, om, os_ = ora.compress_abi(inputs.bf16_bits(W), 1, 512)
    assert np.array_equal(host_bits(gv).ravel(), ov) and np.array_equal(host_bits(gm).ravel(), om)


@pytest.mark.parametrize("gK", [None, 128])
@pytest.mark.parametrize("name", ["tiny", "llama", "groupwise"])
def test_quantize_act_bit_exact(ora, sp24, name, gK):
    w = inputs.WORKLOADS[name]
    X, _, _, _ = inputs.generate(inputs.with_shape(w, N=8))
    gk = w.K if gK is None else gK
    oq, osx = ora.quantize_act(X.numpy(), gk)
    gq, gsx = sp24.quantize_act(dev(X.numpy()), gk)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(gsx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(host_bits(gq), oq)


@pytest.mark.parametrize("gK", [None, 128])
@pytest.mark.parametrize("M,K", [(1, 128), (7, 512), (300, 4096), (513, 384), (2048, 4096), (3000, 4096),
                                 (8192, 4096)])
def test_quantize_act_bf16_bit_exact(ora, sp24, M, K, gK):
    """bf16 activations (the inference dtype of the pages' models): quantized
    exactly as their fp32 widening, which the oracle quantizes.  Rows of
    zeros, bf16 subnormals and values near the bf16 maximum included.  K =
    384 ends each row with a half step of 128 elements; 3000 and 8192 rows of
    4096 take more than one wave of row CTAs."""
    g = torch.Generator().manual_seed(M + K)
    X = (torch.randn(M, K, generator=g) * 3.0).to(torch.bfloat16)
    X[0, :64] = 0.0
    if M > 2:
        X[1] = 0.0                                    # an all-zero row: scale 1.0
        X[2, :8] = torch.tensor([1e-39, -1e-39, 3e-40, 3.3e38, -3.3e38, 1e-38, 0.0, -0.0]).to(torch.bfloat16)
    gk = K if gK is None else gK
    oq, osx = ora.quantize_act(ora.bf16_bits_to_f32(inputs.bf16_bits(X)), gk)
    gq, gsx = sp24.quantize_act(X.cuda(), gk)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(gsx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(host_bits(gq), oq)


def test_quantize_act_bf16_strided_rows(ora, sp24):
    """A bf16 view with a row stride larger than K (a slice of a wider tensor)."""
    g = torch.Generator().manual_seed(9)
    big = torch.randn(40, 768, generator=g).to(torch.bfloat16)
    X = big[:, :512]
    oq, osx = ora.quantize_act(ora.bf16_bits_to_f32(inputs.bf16_bits(X.contiguous())), 128)
    gq, gsx = sp24.quantize_act(big.cuda()[:, :512], 128)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(gsx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(host_bits(gq), oq)


def test_e4m3_rounding_boundaries_on_gpu(ora, sp24):
    """Rows whose amax is 448 have scale exactly 1, so the GPU's e4m3 cast is
    seen directly: every code value, every midpoint and one ulp either side,
    both signs, must round as the oracle's encoder does."""
    q = np.arange(0x7F, dtype=np.uint8)
    v = ora.e4m3_decode(q).astype(np.float32)
    mids = ((v[:-1].astype(np.float64) + v[1:]) / 2).astype(np.float32)
    pts = np.concatenate([v, mids])
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(-np.inf))])
    pts = pts[(np.abs(pts) <= 448)]
    pts = np.concatenate([pts, -pts])
    K = 128
    per_row = K - 1
    rows = (pts.size + per_row - 1) // per_row
    X = np.zeros((rows, K), dtype=np.float32)
    flat = np.zeros(rows * per_row, dtype=np.float32)
    flat[:pts.size] = pts
    X[:, 1:] = flat.reshape(rows, per_row)
    X[:, 0] = 448.0
    oq, osx = ora.quantize_act(X, K)
    gq, gsx = sp24.quantize_act(dev(X), K)
    torch.cuda.synchronize()
    assert (osx == 1.0).all()
    assert np.array_equal(host_bits(gq), oq)


def test_quotients_near_e4m3_midpoints(ora, sp24):
    """Random per-row scales with values placed so that x / s lands on, and a
    few fp32 ulps around, every e4m3 rounding midpoint: the device's division
    (reciprocal with a correction step, exact division near midpoints) must
    give the oracle's correctly rounded codes everywhere."""
    rng = np.random.default_rng(17)
    q = np.arange(0x7F, dtype=np.uint8)
    v = ora.e4m3_decode(q)
    mids = (v[:-1] + v[1:]) / 2                       # includes the subnormal range
    K = 512
    rows = []
    for _ in range(64):
        amax = np.float32(rng.uniform(0.25, 16.0))
        s = np.float32(amax / np.float32(448.0))
        t = rng.choice(mids, size=K - 1) * (1.0 + rng.integers(-4, 5, size=K - 1) * 2.0 ** -23)
        x = (t * np.float64(s)).astype(np.float32) * rng.choice([-1.0, 1.0], size=K - 1).astype(np.float32)
        x = np.clip(x, -amax, amax)
        rows.append(np.concatenate([[amax], x]).astype(np.float32))
    X = np.stack(rows)
    oq, osx = ora.quantize_act(X)
    gq, gsx = sp24.quantize_act(dev(X))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(gsx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(host_bits(gq), oq)
    # the same through weight compression (bf16 rows, kept elements divided by the row scale)
    Wt = torch.from_numpy(X[:, :K].copy()).to(torch.bfloat16)
    Wt = torch.cat([Wt, Wt.flip(0)], 0)               # 128 rows
    ov, om, os_ = ora.compress_abi(inputs.bf16_bits(Wt))
    gv, gm, gs = sp24.compress(dev(inputs.bf16_bits(Wt)))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(gv).ravel(), ov) and np.array_equal(host_bits(gm).ravel(), om)


def test_every_bf16_magnitude_against_many_scales(ora, sp24):
    """Every finite positive bf16 magnitude up to the row's amax is divided by
    that row's scale and rounded to e4m3, for 48 amax values (random, powers of
    two, all-ones mantissas, bf16 subnormal and near the bf16 maximum): the
    device's division must give the oracle's correctly rounded fp32 quotient
    wherever that decides the e4m3 code.  Each group of four is [x, x', 0, 0],
    so both nonzero elements are kept; random signs."""
    rng = np.random.default_rng(23)
    amaxes = [0x3F80, 0x4000, 0x43E0, 0x3FFF, 0x407F, 0x0005, 0x0080, 0x7F7F, 0x7F00, 0x2000, 0x5F7F, 0x3C01]
    amaxes += [int(b) for b in rng.integers(0x0100, 0x7F00, size=36)]
    K = 4096
    rows = []
    for a in amaxes:
        mags = np.arange(1, a + 1, dtype=np.uint32)
        mags = mags[(mags & 0x7F80) != 0x7F80]            # finite only
        per_row = K // 2 - 2                                # group 0 holds [amax, x, 0, 0]
        for start in range(0, len(mags), per_row):
            chunk = mags[start:start + per_row]
            row = np.zeros(K, np.uint16)
            row[0] = a
            xs = np.concatenate([chunk, np.zeros(per_row + 1 - len(chunk), np.uint32)])
            row[1] = xs[0]
            g = xs[1:].reshape(-1, 2)
            body = row[4:].reshape(-1, 4)
            body[:len(g), 0] = g[:, 0]
            body[:len(g), 1] = g[:, 1]
            signs = rng.integers(0, 2, size=K).astype(np.uint16) << 15
            rows.append((row | signs) * (row != 0))
    while len(rows) % 128:
        rows.append(rows[-1])
    Wb = np.stack(rows).astype(np.uint16)
    ov, om, os_ = ora.compress_abi(Wb)
    gv, gm, gs = sp24.compress(dev(Wb))
    torch.cuda.synchronize()
    sp24.last_device_error()
    assert np.array_equal(host_bits(gs).view(np.uint32), os_.view(np.uint32)), "scales"
    assert np.array_equal(host_bits(gm).ravel(), om), "metadata"
    gvb = host_bits(gv).ravel()
    bad = np.flatnonzero(gvb != ov)
    assert bad.size == 0, "%d value bytes differ, first at %s" % (bad.size, bad[:8])


@pytest.mark.parametrize("gN,gK", [(1, None), (1, 128), (128, 128)])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 640), (384, 2176), (1024, 4096)])
def test_decompress_bit_exact(ora, sp24, N, K, gN, gK):
    """GPU dequantize (the dense weight bf16(sw * e4m3) with zeros at the
    pruned positions) from the GPU's own compression: bit-exact against the
    oracle's dequantize of the oracle's compression.  K values that are not
    a multiple of 1024 leave part of the last column of warps idle."""
    g = torch.Generator().manual_seed(N + K)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    gk = K if gK is None else gK
    v, m, s = sp24.compress(W.cuda(), gN, gk)
    D = sp24.decompress(v, m, s, gN, gk)
    torch.cuda.synchronize()
    sp24.last_device_error()
    ov, om, os_ = ora.compress(inputs.bf16_bits(W), gN, gk)
    assert np.array_equal(host_bits(D), ora.dequantize(ov, om, os_, gN, gk))


def test_decompress_strided_output_and_zero_weight(ora, sp24):
    """Output rows wider than K (a view into a larger buffer; the columns
    past K untouched), and an all-zero weight (scale 1, every output +0)."""
    N, K = 256, 512
    g = torch.Generator().manual_seed(4)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    W[:128] = 0.0
    v, m, s = sp24.compress(W.cuda())
    big = torch.full((N, K + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    sp24.decompress(v, m, s, out=big[:, :K])
    torch.cuda.synchronize()
    sp24.last_device_error()
    ov, om, os_ = ora.compress(inputs.bf16_bits(W))
    ref = ora.dequantize(ov, om, os_)
    assert np.array_equal(host_bits(big[:, :K].contiguous()), ref)
    assert np.all(host_bits(big[:, :K].contiguous())[:128] == 0)
    assert torch.all(big[:, K:] == 7.0)
