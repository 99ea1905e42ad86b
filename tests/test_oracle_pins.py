"""Pins for the CPU oracle: each test checks it against something other than
itself -- hand-derived fixtures, a library routine (torch's float8_e4m3fn cast,
numpy matmul), closed forms, invariants, or brute force on tiny inputs.

Chosen so that a plausible slip anywhere in the oracle (a dropped term, a wrong
sign or index, a transposed operand, a flipped tie rule, a wrong rounding mode)
fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _bf16_bits_from_f32(x) -> np.ndarray:
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return inputs.bf16_bits(t)


# ------------------------------------------------------------------ e4m3 codec
def test_e4m3_golden_codes(ora):
    """Hand-derived encodings from the OCP E4M3 definition (fixture file)."""
    vals, codes = [], []
    for line in open(os.path.join(GOLDEN, "e4m3_codes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v, c = line.split()[:2]
        vals.append(float(v))
        codes.append(int(c, 16))
    got = ora.e4m3_encode(np.array(vals, dtype=np.float32))
    assert got.tolist() == codes


def test_e4m3_decode_matches_torch_all_codes(ora):
    """All 256 codes decode like torch's float8_e4m3fn -> float32 conversion."""
    q = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = ora.e4m3_decode(q)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, got[0x80]) == -1.0


def test_e4m3_encode_matches_torch_boundaries(ora):
    """Every finite code value, every midpoint between neighbours, and one fp32
    ulp either side, for both signs; compared with torch's RNE cast (inside
    the range where torch does not overflow, |x| < 464)."""
    q = np.arange(0x7F, dtype=np.uint8)
    v = ora.e4m3_decode(q).astype(np.float32)
    mids = ((v[:-1].astype(np.float64) + v[1:]) / 2).astype(np.float32)
    pts = np.concatenate([v, mids])
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    allp = np.concatenate([pts, up, dn])
    allp = allp[np.abs(allp) < 464]
    allp = np.concatenate([allp, -allp])
    assert np.array_equal(ora.e4m3_encode(allp), _torch_e4m3_bits(allp))


def test_e4m3_encode_matches_torch_random(ora):
    rng = np.random.default_rng(1234)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 50,
        (rng.uniform(-1, 1, 100_000) * 2.0 ** -6).astype(np.float32),   # subnormal range
        rng.uniform(-463.9, 463.9, 100_000).astype(np.float32),
    ])
    assert np.array_equal(ora.e4m3_encode(x), _torch_e4m3_bits(x))


def test_e4m3_saturation_closed_form(ora):
    """Beyond the overflow midpoint the result is the largest finite code."""
    x = np.array([464, 465, 1e4, 3.4e38, -464, -1e30], dtype=np.float32)
    assert ora.e4m3_encode(x).tolist() == [0x7E] * 4 + [0xFE] * 2


def test_e4m3_roundtrip_all_finite_codes(ora):
    q = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert np.array_equal(ora.e4m3_encode(ora.e4m3_decode(q).astype(np.float32)), q)


# ----------------------------------------------------------------------- prune
def test_prune_golden_groups(ora):
    for line in open(os.path.join(GOLDEN, "prune_groups.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        v = _bf16_bits_from_f32([float(t) for t in f[:4]])
        assert ora.keep2(v) == (int(f[4]), int(f[5])), line


def test_prune_bruteforce_all_tuples(ora):
    """Every 4-tuple over a 9-value set (ties, both zeros, both signs):
    the kept pair equals the first two of the positions sorted by
    (descending |v|, ascending index) -- a sort, not the oracle's rank count."""
    vals = [0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0, 3.0]
    bits = dict(zip(vals, _bf16_bits_from_f32(vals).tolist()))
    for tup in itertools.product(vals, repeat=4):
        order = sorted(range(4), key=lambda i: (-abs(tup[i]), i))
        want = tuple(sorted(order[:2]))
        got = ora.keep2(np.array([bits[t] for t in tup], dtype=np.uint16))
        assert got == want, tup


def test_prune_invariants_random(ora):
    w = inputs.with_shape(inputs.WORKLOADS["tiny"], N=64, K=256)
    _, W, _, _ = inputs.generate(w)
    Wb = inputs.bf16_bits(W)
    P = ora.prune(Wb)
    Wf = ora.bf16_bits_to_f32(Wb).reshape(64, -1, 4)
    Pf = ora.bf16_bits_to_f32(P).reshape(64, -1, 4)
    # at most 2 nonzeros per group of 4, and exactly 2 kept positions
    assert ((Pf != 0).sum(-1) <= 2).all()
    # the kept values are the two largest magnitudes
    top2 = -np.sort(-np.abs(Wf), axis=-1)[..., :2]
    kept = -np.sort(-np.abs(Pf), axis=-1)[..., :2]
    assert np.array_equal(top2, kept)
    # group maxima (and so row / block amax) survive pruning
    assert np.array_equal(np.abs(Wf).max(-1), np.abs(Pf).max(-1))


# ---------------------------------------------------------------------- scales
@pytest.mark.parametrize("gN,gK", [(1, None), (1, 128), (128, 128)])
def test_weight_scales_closed_form(ora, gN, gK):
    w = inputs.with_shape(inputs.WORKLOADS["tiny"], N=256, K=512)
    _, W, _, _ = inputs.generate(w)
    Wb = inputs.bf16_bits(W)
    Wf = np.abs(ora.bf16_bits_to_f32(Wb)).reshape(256, 512)
    gk = 512 if gK is None else gK
    s = ora.weight_scales(Wb, gN, gk)
    for kb in range(512 // gk):
        for ng in range(256 // gN):
            amax = np.float32(Wf[ng * gN:(ng + 1) * gN, kb * gk:(kb + 1) * gk].max())
            assert s[kb, ng] == np.float32(amax / np.float32(448.0))


def test_all_zero_weight(ora):
    """All-zero weights must be accepted (torchao PR #3258, jcaip's review of
    the all-zero check): scale 1, codes 0, every group keeps (0, 1)."""
    Wb = np.zeros((16, 256), dtype=np.uint16)
    v, m, s = ora.compress(Wb)
    assert (s == 1.0).all() and (v == 0).all() and (m == 0x44).all()


# --------------------------------------------------- compress / decompress
@pytest.mark.parametrize("gN,gK", [(1, None), (1, 128), (128, 128)])
def test_compress_roundtrip_vs_torch(ora, gN, gK):
    """decompress(compress(W)) equals torch's e4m3 cast of (pruned W / scale),
    bit for bit; the pruned mask and the scales come from independent code."""
    N, K = 256, 512
    w = inputs.with_shape(inputs.WORKLOADS["tiny"], N=N, K=K, seed=7)
    _, W, _, _ = inputs.generate(w)
    Wb = inputs.bf16_bits(W)
    gk = K if gK is None else gK
    values, meta, scales = ora.compress(Wb, gN, gk)
    dense = ora.decompress(values, meta)
    # independent: mask from a numpy sort of |w| per group, scale from numpy amax
    Wf = ora.bf16_bits_to_f32(Wb).reshape(N, K)
    grp = np.abs(Wf).reshape(N, K // 4, 4)
    order = np.argsort(-grp, axis=-1, kind="stable")[..., :2]
    mask = np.zeros_like(grp, dtype=bool)
    np.put_along_axis(mask, order, True, axis=-1)
    pruned = np.where(mask.reshape(N, K), Wf, np.float32(0))
    s_full = np.empty((N, K), dtype=np.float32)
    for kb in range(K // gk):
        for ng in range(N // gN):
            blk = np.abs(Wf[ng * gN:(ng + 1) * gN, kb * gk:(kb + 1) * gk])
            s_full[ng * gN:(ng + 1) * gN, kb * gk:(kb + 1) * gk] = np.float32(blk.max()) / np.float32(448)
    ref = _torch_e4m3_bits(pruned / s_full)
    ref[~mask.reshape(N, K)] = 0  # dropped positions are +0
    assert np.array_equal(dense, ref)
    # at most 2 nonzero codes per group
    assert (((dense.reshape(N, K // 4, 4) & 0x7F) != 0).sum(-1) <= 2).all()


def test_meta_nibbles_are_valid(ora):
    _, W, _, _ = inputs.generate(inputs.with_shape(inputs.WORKLOADS["tiny"], N=32, K=256))
    _, meta, _ = ora.compress(inputs.bf16_bits(W))
    nib = np.stack([meta & 0xF, meta >> 4], -1).ravel()
    i0, i1 = nib & 3, nib >> 2
    assert (i0 < i1).all()


# ------------------------------------------------------------------------ GEMM
def _dense_ref(ora, xq, sx, values, meta, sw, gM, gN, gK, X2=None, W2=None):
    """numpy matmul per K block on the decompressed weight, in float64."""
    M, K = xq.shape
    N = values.shape[0]
    Xd = ora.e4m3_decode(xq)
    Wd = ora.e4m3_decode(ora.decompress(values, meta))
    Y = np.zeros((M, N))
    for kb in range(K // gK):
        sl = slice(kb * gK, (kb + 1) * gK)
        P = Xd[:, sl] @ Wd[:, sl].T
        sxm = np.repeat(sx[kb].astype(np.float64), gM)[:M]
        swn = np.repeat(sw[kb].astype(np.float64), gN)[:N]
        Y += sxm[:, None] * swn[None, :] * P
    if X2 is not None:
        Y += ora.bf16_bits_to_f32(X2).astype(np.float64) @ ora.bf16_bits_to_f32(W2).astype(np.float64).T
    return Y


def _problem(ora, M, N, K, gM, gN, gK, seed, r=0):
    w = inputs.Workload("t", M, N, K, gM=gM, gN=gN, gK=gK, r=r, seed=seed)
    X, W, X2, W2 = inputs.generate(w)
    gk = w.gk
    xq, sx1 = ora.quantize_act(X.numpy(), gk)  # per token (gM = 1)
    if gM != 1:  # coarser activation scales: random positive per block
        rng = np.random.default_rng(seed)
        sx1 = rng.uniform(0.5, 2.0, (K // gk, (M + gM - 1) // gM)).astype(np.float32)
    values, meta, sw = ora.compress(inputs.bf16_bits(W), gN, gk)
    x2 = inputs.bf16_bits(X2) if r else None
    w2 = inputs.bf16_bits(W2) if r else None
    return xq, sx1, values, meta, sw, gk, x2, w2


@pytest.mark.parametrize("gM,gN,gK", [(1, 1, None), (1, 128, 128), (1, 1, 128), (128, 128, 128), (128, 1, None)])
def test_sparse_gemm_equals_dense_gemm(ora, gM, gN, gK):
    """Sparse loop over kept weights == dense matmul on the decompressed W."""
    M, N, K = 130, 256, 512
    xq, sx, v, m, sw, gk, _, _ = _problem(ora, M, N, K, gM, gN, gK, seed=11)
    Y = ora.gemm(xq, sx, v, m, sw, gM, gN, gk, acc_fp64=True)
    ref = _dense_ref(ora, xq, sx, v, m, sw, gM, gN, gk)
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_transpose_identity(ora):
    """C^T = B^T A^T (CUTLASS #2029, klevzoff's swap+transpose answer): the
    oracle's Y[M,N] equals the transpose of W X^T computed with W as the
    left operand."""
    M, N, K = 40, 128, 256
    xq, sx, v, m, sw, gk, _, _ = _problem(ora, M, N, K, 1, 1, None, seed=5)
    Y = ora.gemm(xq, sx, v, m, sw, acc_fp64=True)
    Wd = ora.e4m3_decode(ora.decompress(v, m)) * sw[0][:, None]
    Xd = ora.e4m3_decode(xq) * sx[0][:, None]
    YT = Wd @ Xd.T
    assert np.allclose(Y, YT.T, rtol=1e-12, atol=1e-14)
    assert not np.allclose(Y[:, :M], YT[:M, :], rtol=1e-3)  # and it is not symmetric by accident


def test_granularities_agree_with_unit_scales(ora):
    """CUTLASS PR #2095's 1Dx1D / 1Dx2D / 2Dx1D / 2Dx2D modes: with every scale
    equal to 1 all granularities give the same Y (up to fp32 summation order)."""
    M, N, K = 64, 256, 512
    xq, _, v, m, _, _, _, _ = _problem(ora, M, N, K, 1, 1, None, seed=3)
    outs = []
    for gM in (1, 128):
        for gN in (1, 128):
            for gK in (K, 128):
                sx = np.ones((K // gK, (M + gM - 1) // gM), np.float32)
                sw = np.ones((K // gK, (N + gN - 1) // gN), np.float32)
                outs.append(ora.gemm(xq, sx, v, m, sw, gM, gN, gK))
    for o in outs[1:]:
        assert np.allclose(o, outs[0], rtol=1e-5, atol=1e-4)


def test_bruteforce_tiny(ora):
    """Pure-Python definition on tiny shapes (dense loop over every k, Python
    floats) against the oracle's sparse loop in double."""
    M, N, K, gK = 3, 8, 256, 128
    xq, sx, v, m, sw, gk, _, _ = _problem(ora, M, N, K, 1, 1, gK, seed=9)
    dense = ora.decompress(v, m)
    table = ora.e4m3_decode(np.arange(256, dtype=np.uint8))
    Y = ora.gemm(xq, sx, v, m, sw, 1, 1, gk, acc_fp64=True)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for kb in range(K // gk):
                p = 0.0
                for k in range(kb * gk, (kb + 1) * gk):
                    p += float(table[xq[i, k]]) * float(table[dense[j, k]])
                acc += float(sx[kb, i]) * float(sw[kb, j]) * p
            assert abs(acc - Y[i, j]) <= 1e-12 * max(1.0, abs(acc))


def test_side_gemm(ora):
    """Y = X1 W1^T + X2 W2^T in one result (CUTLASS #2058, hyx1999's shapes,
    scaled down): oracle vs numpy on the two parts."""
    M, N, K, r = 48, 128, 256, 64
    xq, sx, v, m, sw, gk, x2, w2 = _problem(ora, M, N, K, 1, 1, None, seed=6, r=r)
    Y = ora.gemm(xq, sx, v, m, sw, X2=x2, W2=w2, acc_fp64=True)
    ref = _dense_ref(ora, xq, sx, v, m, sw, 1, 1, gk, x2, w2)
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    Y0 = ora.gemm(xq, sx, v, m, sw, acc_fp64=True)
    assert not np.allclose(Y, Y0, rtol=1e-3, atol=1e-3)  # the side term matters


def test_bias_is_added_per_channel(ora):
    """The linear operation's bias (pytorch/ao PR #3258: input, weight, bias):
    with an all-zero weight Y[m, n] is bias[n] exactly in both accumulation
    modes; with a weight, the fp64 result moves by exactly bias[n] (half-integer
    biases on a problem of unit scales and integer products, so that every sum
    is exact in double), column by column, never by row."""
    M, N, K = 8, 128, 256
    bias_f = np.array([(j % 17) - 8 for j in range(N)], dtype=np.float32) * 0.5
    bias = _bf16_bits_from_f32(bias_f)
    v0, m0, sw0 = ora.compress(np.zeros((N, K), np.uint16))
    xq = np.full((M, K), 0x38, np.uint8)  # 1.0
    sx = np.ones((1, M), np.float32)
    for acc64 in (False, True):
        Y = ora.gemm(xq, sx, v0, m0, sw0, bias=bias, acc_fp64=acc64)
        assert np.array_equal(Y, np.broadcast_to(bias_f.astype(np.float64), (M, N)))
    # small integer weights (e4m3 codes of 1 and 2) with unit weight scales
    rng = np.random.default_rng(3)
    Wf = rng.choice([-2.0, -1.0, 0.0, 1.0, 2.0], size=(N, K)).astype(np.float32)
    v, m, _ = ora.compress(_bf16_bits_from_f32(Wf))
    sw = np.ones((1, N), np.float32)
    Y0 = ora.gemm(xq, sx, v, m, sw, acc_fp64=True)
    Yb = ora.gemm(xq, sx, v, m, sw, bias=bias, acc_fp64=True)
    assert np.array_equal(Yb - Y0, np.broadcast_to(bias_f.astype(np.float64), (M, N)))
    assert np.all(Y0 == np.round(Y0))  # the products and sums above are exact integers


def test_f32_to_bf16_matches_torch(ora):
    """Round to nearest even, from fp32 to bf16: against torch's cast on
    random values, exact ties and the values next to them."""
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.normal(0, 1, 4096), rng.normal(0, 1e-30, 256), rng.normal(0, 1e30, 256)])
    ties = (np.arange(1, 513, dtype=np.uint32) << 16) | 0x8000  # exactly halfway, odd and even kept LSB
    near = np.concatenate([ties - 1, ties + 1])
    x = np.concatenate([x.astype(np.float32), ties.view(np.float32), near.view(np.float32),
                        np.array([0.0, -0.0, 3.3e38, -3.3e38], np.float32)])
    ref = inputs.bf16_bits(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(ora.f32_to_bf16_bits(x), ref)


@pytest.mark.parametrize("gN,gK", [(1, None), (1, 128), (128, 128)])
def test_dequantize_is_the_identity_gemm(ora, gN, gK):
    """Dequantize = the GEMM of an identity activation with unit scales,
    rounded to bf16 by torch (pytorch/ao PR #3258, dequantize by multiplying
    with an identity); +0 exactly where the metadata drops a weight."""
    N, K = 128, 256
    _, W, _, _ = inputs.generate(inputs.with_shape(inputs.WORKLOADS["tiny"], N=N, K=K, seed=8))
    v, m, sw = ora.compress(inputs.bf16_bits(W), gN, gK)
    gk = K if gK is None else gK
    D = ora.dequantize(v, m, sw, gN, gk)
    xq = np.where(np.eye(K, dtype=bool), 0x38, 0).astype(np.uint8)
    sx = np.ones((K // gk, K), np.float32)
    Y = ora.gemm(xq, sx, v, m, sw, 1, gN, gk)                  # [K tokens, N channels]
    ref = inputs.bf16_bits(torch.from_numpy(Y.astype(np.float32).T.copy()).to(torch.bfloat16))
    assert np.array_equal(D, ref)
    assert np.all(D[ora.decompress(v, m) == 0] == 0)
    assert np.count_nonzero(ora.decompress(v, m)) <= N * K // 2


def test_identity_dequantize(ora):
    """Dequantize by multiplying with an identity (torchao PR #3258, jcaip's
    review of dequantize): X = I (code 0x38 = 1.0), unit activation scales
    -> Y[k, n] = sw[n] * Wq[n, k] exactly."""
    N, K = 64, 256
    _, W, _, _ = inputs.generate(inputs.with_shape(inputs.WORKLOADS["tiny"], N=N, K=K, seed=2))
    v, m, sw = ora.compress(inputs.bf16_bits(W))
    xq = np.where(np.eye(K, dtype=bool), 0x38, 0).astype(np.uint8)
    sx = np.ones((1, K), np.float32)
    Y = ora.gemm(xq, sx, v, m, sw)
    Wq = ora.e4m3_decode(ora.decompress(v, m))
    ref = (Wq * sw[0][:, None].astype(np.float64)).astype(np.float32).T
    assert np.array_equal(Y.astype(np.float32), ref)


def test_fp32_accumulation_error_bound(ora):
    """The fp32-accumulated oracle stays within the standard summation bound
    of the double one: |d| <= n * 2^-24 * sum|terms| (n terms)."""
    M, N, K = 32, 128, 1024
    xq, sx, v, m, sw, gk, _, _ = _problem(ora, M, N, K, 1, 128, 128, seed=4)
    Y32 = ora.gemm(xq, sx, v, m, sw, 1, 128, 128)
    Y64 = ora.gemm(xq, sx, v, m, sw, 1, 128, 128, acc_fp64=True)
    Xd = np.abs(ora.e4m3_decode(xq))
    Wd = np.abs(ora.e4m3_decode(ora.decompress(v, m)))
    absum = np.zeros((M, N))
    for kb in range(K // 128):
        sl = slice(kb * 128, (kb + 1) * 128)
        absum += np.outer(sx[kb], np.repeat(sw[kb], 128)) * (Xd[:, sl] @ Wd[:, sl].T)
    n = K // 2 + 2 * (K // 128) + 2
    assert (np.abs(Y32 - Y64) <= n * 2.0 ** -24 * absum + 1e-30).all()


# --------------------------------------------------- activation quantization
@pytest.mark.parametrize("gK", [None, 128])
def test_quantize_act_closed_form(ora, gK):
    X, _, _, _ = inputs.generate(inputs.with_shape(inputs.WORKLOADS["llama"], M=64, N=16, K=512))
    Xn = X.numpy()
    gk = 512 if gK is None else gK
    xq, sx = ora.quantize_act(Xn, gk)
    for kb in range(512 // gk):
        blk = Xn[:, kb * gk:(kb + 1) * gk]
        s = (np.abs(blk).max(1).astype(np.float32) / np.float32(448)).astype(np.float32)
        assert np.array_equal(sx[kb], s)
        assert np.array_equal(xq[:, kb * gk:(kb + 1) * gk], _torch_e4m3_bits(blk / s[:, None]))


def test_oracle_shares_nothing_with_cuda_path():
    """The oracle and the CUDA package never import or include each other."""
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    bad_in_oracle = re.compile(r"(import|from)\s+semi_structured_sparse_gb300|#include\s+[<\"].*sp24")
    for dirpath, _, files in os.walk(os.path.join(root, "oracle")):
        for f in files:
            if f.endswith((".py", ".c", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert not bad_in_oracle.search(txt), f
    bad_in_pkg = re.compile(r"(import|from)\s+oracle|sp24_oracle|liboracle")
    for dirpath, _, files in os.walk(os.path.join(root, "semi_structured_sparse_gb300")):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert not bad_in_pkg.search(txt), f


# --------------------------------------------------------- storage layout
def test_tiled_layout_is_a_permutation(ora):
    N, K = 256, 512
    rng = np.random.default_rng(0)
    v = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    m = rng.integers(0, 256, (N, K // 8), dtype=np.uint8)
    tv, tm = ora.tile_values(v), ora.tile_meta(m)
    assert np.array_equal(ora.untile_values(tv, N, K), v)
    assert np.array_equal(ora.untile_meta(tm, N, K), m)
    # distinct positions: tile an index pattern and check every slot is hit once
    idx = np.arange(N * K // 2, dtype=np.int64)
    hit = np.zeros(N * K // 2, dtype=np.int64)
    for shift in (0, 8, 16):
        t = ora.tile_values(((idx >> shift) & 0xFF).astype(np.uint8).reshape(N, K // 2))
        hit += t.astype(np.int64) << shift
    assert np.array_equal(np.sort(hit), idx)


def test_tiled_layout_known_positions(ora):
    """Hand-computed positions: tile (n-band, k-block) order, row pitch 64 B,
    16-byte chunks XOR-swizzled with (row/2) mod 4; metadata rows of 16 B."""
    N, K = 256, 512
    v = np.zeros((N, K // 2), np.uint8)
    v[0, 0] = 1        # tile 0, row 0, chunk 0 -> offset 0
    v[2, 0] = 2        # row 2: chunk 0 ^ 1 = 1 -> 2*64 + 16 = 144
    v[7, 17] = 3       # row 7: (7//2)%4 = 3, chunk 1 ^ 3 = 2 -> 7*64 + 32 + 1 = 481
    v[0, 64] = 4       # second K tile of band 0 -> 8192
    v[130, 70] = 5     # band 1 (tiles 4..7), k tile 1 -> tile 5; row 2, b 6, chunk 0^1 -> 5*8192 + 128 + 16 + 6
    t = ora.tile_values(v)
    assert t[0] == 1 and t[144] == 2 and t[481] == 3 and t[8192] == 4 and t[5 * 8192 + 150] == 5
    m = np.zeros((N, K // 8), np.uint8)
    m[1, 3] = 7        # tile 0: 1*16 + 3
    m[129, 20] = 9     # band 1, k tile 1 -> tile 5: 1*16 + 4
    tm = ora.tile_meta(m)
    assert tm[19] == 7 and tm[5 * 2048 + 20] == 9


# ---------------------------------------------------------------- int8 sibling
def test_int8_rounding_golden(ora):
    """Hand-derived: ties go to the even integer, both signs; the clamp."""
    cases = {2.5: 2, 3.5: 4, -2.5: -2, -3.5: -4, 0.5: 0, -0.5: 0, 1.5: 2, 126.5: 126, 125.5: 126,
             127.4: 127, 127.5: 127, 200.0: 127, -300.0: -127, 0.49999997: 0, 2.5000002: 3, -0.0: 0}
    for x, q in cases.items():
        assert ora.int8_encode(x) == q, x


def test_int8_rounding_matches_numpy(ora):
    """numpy's rint (round half to even) on fp32 grids: every half point in
    [-128, 128], its fp32 neighbours, and random values."""
    rng = np.random.default_rng(8)
    half = np.arange(-256, 257, dtype=np.float32) / 2
    grid = np.concatenate([half, np.nextafter(half, np.float32(np.inf)), np.nextafter(half, np.float32(-np.inf)),
                           rng.uniform(-127, 127, 3000).astype(np.float32)])
    want = np.clip(np.rint(grid.astype(np.float64)), -127, 127).astype(np.int64)
    got = np.array([ora.int8_encode(x) for x in grid])
    assert np.array_equal(got, want)


def test_int8_compress_against_numpy(ora):
    """Per-channel scale = amax/127 and q = rint(fp32(w / s)) computed with
    numpy's fp32 division; the pruning and metadata are the FP8 weight's."""
    w = inputs.Workload("i8c", 1, 256, 512, seed=17)
    _, W, _, _ = inputs.generate(w)
    bits = inputs.bf16_bits(W)
    values, meta, scales = ora.compress_int8(bits)
    _, meta_fp8, _ = ora.compress(bits)
    assert np.array_equal(meta, meta_fp8)
    Wf = ora.bf16_bits_to_f32(bits)
    amax = np.abs(Wf).max(axis=1)
    s_np = np.where(amax == 0, np.float32(1), (amax / np.float32(127)).astype(np.float32))
    assert np.array_equal(scales.view(np.uint32), s_np.astype(np.float32).view(np.uint32))
    # the kept values, read through the metadata
    N, K = Wf.shape
    for n in range(0, N, 37):
        for g in range(K // 4):
            nib = (int(meta[n, g // 2]) >> (4 * (g & 1))) & 0xF
            i0, i1 = nib & 3, nib >> 2
            for t, i in enumerate((i0, i1)):
                q = np.rint(np.float64(np.float32(Wf[n, 4 * g + i]) / np.float32(scales[n])))
                assert values[n, 2 * g + t] == int(np.clip(q, -127, 127))
    # the row maximum maps to +-127
    assert np.abs(values.astype(np.int64)).max(axis=1).min() == 127


def test_int8_gemm_equals_integer_matmul(ora):
    """The int32 sums equal numpy's exact int64 matmul of the dense int8
    operands (the kept weights at their positions, zeros elsewhere); Y is the
    fp32 product of the two scales and the sum, plus the bias."""
    rng = np.random.default_rng(9)
    w = inputs.Workload("i8g", 37, 256, 768, seed=19)
    X, W, _, _ = inputs.generate(w)
    values, meta, sw = ora.compress_int8(inputs.bf16_bits(W))
    xq, sx = ora.quantize_act_int8(X.numpy())
    bias = inputs.bf16_bits(torch.from_numpy(rng.normal(size=256).astype(np.float32)).to(torch.bfloat16))
    Y, acc = ora.gemm_int8(xq, sx, values, meta, sw, bias=bias)
    dense = np.zeros((256, 768), dtype=np.int64)
    for g in range(768 // 4):
        nib = (meta[:, g // 2].astype(np.int64) >> (4 * (g & 1))) & 0xF
        rows = np.arange(256)
        dense[rows, 4 * g + (nib & 3)] = values[:, 2 * g]
        dense[rows, 4 * g + (nib >> 2)] = values[:, 2 * g + 1]
    ref = xq.astype(np.int64) @ dense.T
    assert np.array_equal(acc.astype(np.int64), ref)
    y32 = (sx[:, None] * sw[None, :]).astype(np.float32) * ref.astype(np.float32)
    y32 = (y32 + ora.bf16_bits_to_f32(bias)[None, :]).astype(np.float32)
    assert np.array_equal(Y.astype(np.float32), y32)


def test_int8_quantize_act_against_numpy(ora):
    rng = np.random.default_rng(10)
    X = rng.normal(size=(9, 384)).astype(np.float32)
    X[3] = 0.0
    xq, sx = ora.quantize_act_int8(X)
    amax = np.abs(X).max(axis=1)
    s_np = np.where(amax == 0, np.float32(1), (amax / np.float32(127)).astype(np.float32)).astype(np.float32)
    assert np.array_equal(sx, s_np)
    q = np.clip(np.rint((X / s_np[:, None]).astype(np.float32).astype(np.float64)), -127, 127)
    assert np.array_equal(xq.astype(np.int64), q.astype(np.int64))
    assert not xq[3].any()


def test_int8_bruteforce_tiny(ora):
    """A 1 x 8 x 8 case summed by hand in Python integers."""
    W = np.array([[3, -1, 0, 2, 5, 5, -7, 1]] * 8, dtype=np.float32) * np.arange(1, 9, dtype=np.float32)[:, None]
    X = np.array([[1, -2, 3, -4, 5, -6, 7, -8]], dtype=np.float32)
    bits = _bf16_bits_from_f32(W)
    values, meta, sw = ora.compress_int8(bits)
    xq, sx = ora.quantize_act_int8(X)
    _, acc = ora.gemm_int8(xq, sx, values, meta, sw)
    for n in range(8):
        total = 0
        for g in range(2):
            nib = (int(meta[n, 0]) >> (4 * g)) & 0xF
            for t, i in enumerate((nib & 3, nib >> 2)):
                total += int(values[n, 2 * g + t]) * int(xq[0, 4 * g + i])
        assert acc[0, n] == total
        # the two kept of (3, -1, 0, 2) are 3 and 2; of (5, 5, -7, 1), -7 and the first 5
        assert (meta[n, 0] & 0xF) == (0 | 3 << 2) and (meta[n, 0] >> 4) == (0 | 2 << 2)
