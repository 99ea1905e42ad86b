"""GPU parity of the 2:4 sparse FP8 GEMM against the CPU oracle, through the C ABI.

Inputs are the seeded synthetic workloads; both sides consume the same bytes
(the oracle's compression and activation quantization).  Tolerance, element by
element: |Y - ref| <= 1e-2 |ref| + 1e-3 with ref the oracle's fp32-accumulated
result (the bf16 output rounding alone is <= 2^-9 |ref|).

Every test compares every output element: the small cases (several tiles,
ragged token tails, every granularity) and the full-size workloads, run in
the same launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import inputs
from gpu_util import assert_close, bf16_to_f64, dev

pytestmark = pytest.mark.gpu


def _prep(ora, w: inputs.Workload):
    X, W, X2, W2 = inputs.generate(w)
    gk = w.gk
    xq, sx = ora.quantize_act(X.numpy(), gk)
    if w.gM != 1:  # coarser activation scales are caller-supplied: any positive values
        rng = np.random.default_rng(w.seed)
        sx = rng.uniform(0.001, 0.01, (w.K // gk, (w.M + w.gM - 1) // w.gM)).astype(np.float32)
    values, meta, sw = ora.compress(inputs.bf16_bits(W), w.gN, gk)
    x2 = inputs.bf16_bits(X2) if w.r else None
    w2 = inputs.bf16_bits(W2) if w.r else None
    return xq, sx, values, meta, sw, x2, w2


def _abi(ora, values, meta):
    """Logical (values, meta) -> the tiled storage the library reads, as [N, K/2] / [N, K/8]."""
    N = values.shape[0]
    return (ora.tile_values(values).reshape(N, -1), ora.tile_meta(meta).reshape(N, -1))


def _run_gpu(sp24, w, xq, sx, values, meta, sw, x2, w2):
    import oracle as ora
    values, meta = _abi(ora, values, meta)
    y = sp24.gemm(dev(xq), dev(sx), dev(values), dev(meta), dev(sw), w.gM, w.gN, w.gk,
                  None if x2 is None else dev(x2), None if w2 is None else dev(w2))
    torch.cuda.synchronize()
    sp24.last_device_error()
    return bf16_to_f64(y)


def _check_full(ora, sp24, w, what):
    xq, sx, values, meta, sw, x2, w2 = _prep(ora, w)
    y = _run_gpu(sp24, w, xq, sx, values, meta, sw, x2, w2)
    ref = ora.gemm(xq, sx, values, meta, sw, w.gM, w.gN, w.gk, x2, w2)
    assert_close(y, ref, what)
    return y, ref


def test_tiny_workload(ora, sp24):
    w = inputs.WORKLOADS["tiny"]
    y, ref = _check_full(ora, sp24, w, "tiny")
    assert np.abs(ref).max() > 0.1  # the comparison is not vacuous


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32, 33, 64, 65, 128, 129, 300])
def test_token_counts_per_channel(ora, sp24, M):
    w = inputs.Workload("pc", M, 384, 512, seed=100 + M)
    _check_full(ora, sp24, w, "M=%d" % M)


@pytest.mark.parametrize("gM,gN,gK", [(1, 128, 128), (1, 1, 128), (128, 128, 128), (128, 1, None),
                                       (1, 128, None), (128, 1, 128)])
@pytest.mark.parametrize("M", [5, 130, 300])
def test_granularities(ora, sp24, gM, gN, gK, M):
    w = inputs.Workload("g", M, 384, 768, gM=gM, gN=gN, gK=gK, seed=7 * M + gM + gN)
    _check_full(ora, sp24, w, "g=(%d,%d,%s) M=%d" % (gM, gN, gK, M))


@pytest.mark.parametrize("r", [16, 32, 64])
@pytest.mark.parametrize("M,gK", [(40, None), (200, None), (130, 128)])
def test_side_gemm(ora, sp24, r, M, gK):
    w = inputs.Workload("side", M, 256, 512, gK=gK, r=r, seed=r + M)
    _check_full(ora, sp24, w, "side r=%d M=%d" % (r, M))


@pytest.mark.parametrize("M,N,K,gN,gK,r", [
    (40, 384, 512, 1, None, 0),     # one-CTA kernel, 64-token tiles
    (16, 1024, 1024, 1, None, 0),   # decode tiles with K split across CTAs
    (300, 384, 512, 1, None, 0),    # one-CTA 256-token tiles (N not a multiple of 256)
    (300, 512, 512, 1, None, 0),    # SM pairs
    (300, 512, 512, 1, None, 32),   # SM pairs with the side GEMM
    (40, 256, 512, 1, None, 16),    # one-CTA side GEMM
    (130, 384, 768, 128, 128, 0),   # one-CTA group-wise promotion
    (300, 512, 768, 128, 128, 0),   # SM-pair group-wise promotion
    (130, 256, 512, 1, 128, 16),    # promotion with the side GEMM
])
def test_bias(ora, sp24, M, N, K, gN, gK, r):
    """The linear operation's bias (pytorch/ao PR #3258: input, weight, bias),
    added in fp32 before the one rounding to bf16, on every epilogue path."""
    w = inputs.Workload("bias", M, N, K, gN=gN, gK=gK, r=r, seed=M + N + K + r)
    xq, sx, values, meta, sw, x2, w2 = _prep(ora, w)
    rng = np.random.default_rng(w.seed)
    bias = inputs.bf16_bits(torch.from_numpy(rng.normal(0.0, 0.5, N).astype(np.float32)).to(torch.bfloat16))
    tv, tm = _abi(ora, values, meta)
    y = sp24.gemm(dev(xq), dev(sx), dev(tv), dev(tm), dev(sw), w.gM, w.gN, w.gk,
                  None if x2 is None else dev(x2), None if w2 is None else dev(w2), bias=dev(bias))
    torch.cuda.synchronize()
    sp24.last_device_error()
    ref = ora.gemm(xq, sx, values, meta, sw, w.gM, w.gN, w.gk, x2, w2, bias=bias)
    assert_close(bf16_to_f64(y), ref, "bias M=%d N=%d K=%d gK=%s r=%d" % (M, N, K, gK, r))
    assert np.abs(ref - ora.gemm(xq, sx, values, meta, sw, w.gM, w.gN, w.gk, x2, w2)).max() > 0.1


def test_zero_bias_matches_no_bias(ora, sp24):
    """A zero bias gives the values of no bias (the kernels fold -0.0 in when
    there is none, which changes no value; +0.0 may only turn -0.0 into +0.0,
    which compares equal)."""
    w = inputs.Workload("nobias", 300, 512, 512, seed=5)
    xq, sx, values, meta, sw, _, _ = _prep(ora, w)
    tv, tm = _abi(ora, values, meta)
    a = sp24.gemm(dev(xq), dev(sx), dev(tv), dev(tm), dev(sw))
    z = torch.zeros(w.N, dtype=torch.bfloat16, device="cuda")
    b = sp24.gemm(dev(xq), dev(sx), dev(tv), dev(tm), dev(sw), bias=z)
    torch.cuda.synchronize()
    sp24.last_device_error()
    assert np.array_equal(a.float().cpu().numpy(), b.float().cpu().numpy())
    assert_close(bf16_to_f64(a), ora.gemm(xq, sx, values, meta, sw), "no bias")


def test_k_equals_128(ora, sp24):
    _check_full(ora, sp24, inputs.Workload("k128", 70, 128, 128, seed=3), "K=128")
    _check_full(ora, sp24, inputs.Workload("k128g", 70, 128, 128, gN=128, gK=128, seed=4), "K=128 gK=128")


def test_identity_dequantize(ora, sp24):
    """X = I (e4m3 1.0 on the diagonal), unit activation scales: Y[k, n] is the
    dequantized weight sw[n] * Wq[n, k] (pytorch/ao PR #3258, jcaip: dequantize
    by multiplying with an identity), rounded to bf16, exactly."""
    N, K = 256, 512
    _, W, _, _ = inputs.generate(inputs.Workload("id", 1, N, K, seed=21))
    values, meta, sw = ora.compress(inputs.bf16_bits(W))
    xq = np.where(np.eye(K, dtype=bool), 0x38, 0).astype(np.uint8)
    sx = np.ones((1, K), np.float32)
    tv, tm = _abi(ora, values, meta)
    y = sp24.gemm(dev(xq), dev(sx), dev(tv), dev(tm), dev(sw))
    torch.cuda.synchronize()
    Wq = ora.e4m3_decode(ora.decompress(values, meta))
    ref = torch.from_numpy((Wq * sw[0][:, None]).astype(np.float32).T.copy()).to(torch.bfloat16)
    assert torch.equal(y.cpu(), ref)


def test_all_zero_weight(ora, sp24):
    M, N, K = 64, 128, 256
    X, _, _, _ = inputs.generate(inputs.Workload("z", M, N, K, seed=1))
    xq, sx = ora.quantize_act(X.numpy())
    values, meta, sw = ora.compress_abi(np.zeros((N, K), np.uint16))
    y = sp24.gemm(dev(xq), dev(sx), dev(values.reshape(N, -1)), dev(meta.reshape(N, -1)), dev(sw))
    torch.cuda.synchronize()
    assert (y.float() == 0).all()


def test_one_hot_weight_patterns(ora, sp24):
    """Each weight row keeps one nonzero at a known position per group of
    four (and its partner at a zero value): checks that every metadata
    nibble steers the right activation column, end to end."""
    M, N, K = 64, 128, 256
    rng = np.random.default_rng(8)
    Wf = np.zeros((N, K), np.float32)
    pos = rng.integers(0, 4, size=(N, K // 4))
    Wf.reshape(N, K // 4, 4)[np.arange(N)[:, None], np.arange(K // 4)[None, :], pos] = \
        rng.uniform(0.5, 1.5, (N, K // 4)).astype(np.float32)
    Wb = inputs.bf16_bits(torch.from_numpy(Wf).to(torch.bfloat16))
    X, _, _, _ = inputs.generate(inputs.Workload("oh", M, N, K, seed=2))
    xq, sx = ora.quantize_act(X.numpy())
    values, meta, sw = ora.compress(Wb)
    y = _run_gpu(sp24, inputs.Workload("oh", M, N, K), xq, sx, values, meta, sw, None, None)
    ref = ora.gemm(xq, sx, values, meta, sw)
    assert_close(y, ref, "one-hot")


def test_repeat_is_deterministic(ora, sp24):
    w = inputs.Workload("det", 300, 384, 1024, gN=128, gK=128, seed=77)
    xq, sx, values, meta, sw, _, _ = _prep(ora, w)
    values, meta = _abi(ora, values, meta)
    a = [dev(t) for t in (xq, sx, values, meta, sw)]
    y1 = sp24.gemm(*a, w.gM, w.gN, w.gk)
    y2 = sp24.gemm(*a, w.gM, w.gN, w.gk)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


# ------------------------------------------------------------- full-size runs
@pytest.mark.parametrize("name", ["llama", "groupwise", "fused"])
def test_full_size(ora, sp24, name):
    """The full-size workloads, in the launch configuration the benchmark
    times, compared with the oracle on every output element."""
    w = inputs.WORKLOADS[name]
    y, ref = _check_full(ora, sp24, w, name + " (every element)")
    assert y.shape == (w.M, w.N) and np.isfinite(y).all()


@pytest.mark.parametrize("M", inputs.DECODE_M)
def test_decode_full_size(ora, sp24, M):
    """The decode sweep's full-size weight (N 28672, K 4096) at every token
    count of the sweep, every output element."""
    w = inputs.with_shape(inputs.WORKLOADS["decode"], M=M)
    _check_full(ora, sp24, w, "decode M=%d (every element)" % M)


def test_compress_then_gemm_on_device(ora, sp24):
    """The whole path on the device (quantize, compress, GEMM) against the
    whole path in the oracle."""
    w = inputs.with_shape(inputs.WORKLOADS["llama"], M=256, N=512, K=1024)
    X, W, _, _ = inputs.generate(w)
    xq_d, sx_d = sp24.quantize_act(X.cuda())
    v_d, m_d, sw_d = sp24.compress(dev(inputs.bf16_bits(W)))
    y = bf16_to_f64(sp24.gemm(xq_d, sx_d, v_d, m_d, sw_d))
    xq, sx = ora.quantize_act(X.numpy())
    values, meta, sw = ora.compress(inputs.bf16_bits(W))
    assert_close(y, ora.gemm(xq, sx, values, meta, sw), "device path")


# ---------------------------------------------------------------- SM pairs
@pytest.mark.parametrize("M,N,K", [(193, 256, 256), (256, 768, 128), (300, 768, 512), (511, 256, 1024),
                                   (2048, 2816, 256)])
def test_pair_tiles(ora, sp24, M, N, K):
    """More than 192 tokens with N an odd multiple of 256 run on SM pairs:
    one M = 256 sparse MMA across two SMs per 128-wide K half-step, 256 x 256
    output tiles.  Ragged token tails (the second SM's activation rows past
    M), a single K block, and more tiles than pairs (each pair loops)."""
    w = inputs.Workload("pair", M, N, K, seed=M + N + K)
    _check_full(ora, sp24, w, "pair M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(240, 512, 128), (241, 1024, 640), (481, 512, 1024), (1000, 1536, 2048),
                                   (2048, 5120, 256)])
def test_pair_tiles_more_shapes(ora, sp24, M, N, K):
    """More pair-tile shapes: token tails inside the first and second SM's
    halves of a 256-token tile, a single K block, K block counts that are not
    a multiple of the stage depth, and more tiles than pairs (2048 x 5120:
    160 tiles, so pairs store one tile while the next one runs)."""
    w = inputs.Workload("pair2", M, N, K, seed=M + N + K + 1)
    _check_full(ora, sp24, w, "pair M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(512, 19456, 256), (520, 19456, 384), (2048, 4096, 512), (721, 2048, 768)])
def test_pair_token_tiles(ora, sp24, M, N, K):
    """The plain pair kernel's token tile, 256 or 240, whichever takes fewer
    tile-widths of time over the rounds of tiles on the SM pairs.  On a
    152-SM part: 512 x 19456 is 152 tiles of 256 in two rounds (228 of 240
    would take three), so it runs 256-token tiles; 520 tokens need three
    rounds either way (3 x 240 < 3 x 256); 2048 x 4096 is 144 tiles of 240
    in two rounds against 128 of 256, also two; 721 tokens end 1 past a
    240 boundary (a one-token tile in the first SM's half)."""
    w = inputs.Workload("ptile", M, N, K, seed=M + N + K + 2)
    _check_full(ora, sp24, w, "pair token tile M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K,r", [(193, 256, 256, 64), (240, 512, 128, 16), (241, 512, 384, 32),
                                     (481, 768, 1024, 48), (2048, 2816, 256, 64)])
def test_pair_tiles_side_gemm(ora, sp24, M, N, K, r):
    """The fused side GEMM on SM pairs: 240-token tiles with the main and the
    side accumulator side by side in tensor memory, the side operands loaded
    as the first stage of each tile.  Tails in both halves of a tile, a single
    K block, r not a power of two, and more tiles than pairs (99 tiles:
    pairs store one tile while the next one runs)."""
    w = inputs.Workload("pside", M, N, K, r=r, seed=M + N + K + r)
    _check_full(ora, sp24, w, "pair side M=%d N=%d K=%d r=%d" % (M, N, K, r))


@pytest.mark.parametrize("gM,gN", [(1, 128), (1, 1), (128, 128), (128, 1)])
@pytest.mark.parametrize("M,N,K", [(65, 256, 256), (130, 512, 768), (300, 768, 1024), (2000, 1536, 512)])
def test_pair_tiles_groupwise(ora, sp24, gM, gN, M, N, K):
    """Group-wise promotion (gK = 128) on SM pairs: each K block's partial in
    one of the tensor-memory accumulators, scaled by its own sx sw into fp32
    registers.  These shapes take as many rounds of tiles with 112 tokens as
    with 128, so they run the 112-token tiles (four accumulators).
    Per-channel and 128-row block weight scales, per-token and 128-token
    block activation scales, token tails in either SM's half of a tile, a
    single stage, four stages per tile (K = 1024), and more tiles than pairs
    (2000 x 1536: 18 token tiles x 6 weight-row tiles = 108)."""
    w = inputs.Workload("pairgw", M, N, K, gM=gM, gN=gN, gK=128, seed=M + N + K + gM + 3 * gN)
    _check_full(ora, sp24, w, "pair group-wise g=(%d,%d) M=%d N=%d K=%d" % (gM, gN, M, N, K))


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 256), (1000, 4096, 512), (513, 4096, 256), (1024, 14336, 256),
                                   (1100, 14336, 256)])
def test_pair_promote_token_tiles(ora, sp24, M, N, K):
    """The group-wise pair kernel's token tile: 112 (four accumulators) where
    it takes no more rounds of tiles over the SM pairs than 128 (three), else
    128.  On a 152-SM part: 2048 x 4096 is four rounds either way, 1000 and
    513 tokens (a 65-token last tile: 56 in the first SM's half, 9 in the
    second) two, so those run 112; 1024 x 14336 is 6 rounds of 128 against 8
    of 112, and 1100 tokens 7 against 8 (a 76-token last tile), so those run
    128, the tile of the group-wise benchmark."""
    w = inputs.Workload("pgwtile", M, N, K, gN=128, gK=128, seed=M + N + K + 9)
    _check_full(ora, sp24, w, "group-wise pair token tile M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("gM,gN", [(128, 128), (1, 1), (128, 1)])
def test_pair_promote_128_token_tiles_granularities(ora, sp24, gM, gN):
    """The 128-token group-wise tiles (the benchmark's) with the other scale
    granularities: 128-token activation blocks and per-channel weight scales,
    on 1100 x 14336 (7 rounds of 128-token tiles against 8 of 112)."""
    w = inputs.Workload("pgw128", 1100, 14336, 256, gM=gM, gN=gN, gK=128, seed=gM + 5 * gN)
    _check_full(ora, sp24, w, "group-wise 128-token tiles g=(%d,%d)" % (gM, gN))


def test_groupwise_odd_k_blocks_falls_back(ora, sp24):
    """An odd number of 128-wide K blocks does not fill the pair kernel's
    two-block stages: such calls run on the one-CTA kernel, with the same result."""
    w = inputs.Workload("gwodd", 300, 512, 384, gN=128, gK=128, seed=11)
    _check_full(ora, sp24, w, "group-wise odd K blocks")


@pytest.mark.parametrize("gM,gN", [(128, 128), (1, 128), (128, 1)])
def test_pair_tiles_coarse_scales(ora, sp24, gM, gN):
    w = inputs.Workload("pairg", 400, 512, 384, gM=gM, gN=gN, seed=gM + 3 * gN)
    _check_full(ora, sp24, w, "pair gM=%d gN=%d" % (gM, gN))


def test_pair_tiles_deterministic(ora, sp24):
    w = inputs.Workload("pdet", 700, 1024, 512, seed=5)
    xq, sx, values, meta, sw, _, _ = _prep(ora, w)
    values, meta = _abi(ora, values, meta)
    a = [dev(t) for t in (xq, sx, values, meta, sw)]
    y1 = sp24.gemm(*a)
    y2 = sp24.gemm(*a)
    torch.cuda.synchronize()
    sp24.last_device_error()
    assert torch.equal(y1, y2)


# ------------------------------------------------------------------ stream-K
@pytest.mark.parametrize("M,N,K", [(16, 5120, 4096), (1, 5120, 4096), (64, 4096, 4096), (33, 6144, 2048),
                                   (16, 256, 2048),     # fewer work units than SMs: one per CTA
                                   (7, 14336, 4096)])   # about six units per CTA, cut across tiles
def test_split_k(ora, sp24, M, N, K):
    """Stream-K forced on small-token shapes: the (tile, K block) work is dealt
    out in equal ranges, and the CTA holding a tile's first K blocks adds the
    other CTAs' partials in a fixed order."""
    w = inputs.Workload("sk", M, N, K, seed=M + N)
    with sp24.decomposition(sp24.DECOMP_STREAM_K):
        assert sp24.workspace_size(M, N, K) > 0, "this shape is expected to split K"
        y, ref = _check_full(ora, sp24, w, "split-K M=%d N=%d K=%d" % (M, N, K))
        # deterministic: same bits on a second run
        xq, sx, values, meta, sw, _, _ = _prep(ora, w)
        y2 = _run_gpu(sp24, w, xq, sx, values, meta, sw, None, None)
    assert np.array_equal(y, y2)
    # and whole tiles give the same values within rounding
    with sp24.decomposition(sp24.DECOMP_DATA_PARALLEL):
        assert sp24.workspace_size(M, N, K) == 0
        y3 = _run_gpu(sp24, w, xq, sx, values, meta, sw, None, None)
    assert_close(y3, ref, "whole tiles M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K,expect", [
    (16, 4096, 14336, (3, 4)),   # few weight tiles, long K: a cluster of 4 CTAs per tile
    (64, 4096, 14336, (3, 2)),   # 64-token tiles: clusters of 2
    (16, 4096, 4096, (3, 4)),
    (16, 6144, 4096, (3, 2)),    # 48 tiles: clusters of 2 (4 would not fit in one wave)
    (16, 14336, 4096, (1, 1)),   # 112 tiles: no room to split, whole tiles already stream at the HBM rate
    (16, 28672, 4096, (1, 1)),   # enough tiles for whole rounds
    (128, 4096, 14336, (1, 1)),  # 128-token tiles: whole tiles only
])
def test_heuristic_decomposition(sp24, M, N, K, expect):
    """The default mode's choice (cost model on a 152-SM part)."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are those of a 152-SM part")
    assert sp24.decomposition_of(M, N, K) == expect
    assert sp24.workspace_size(M, N, K) == 0


def test_heuristic_split_shape(ora, sp24):
    """A shape the heuristic itself splits, through the default path."""
    M, N, K = 5, 1024, 16384
    assert sp24.decomposition_of(M, N, K)[0] != sp24.DECOMP_DATA_PARALLEL
    w = inputs.Workload("skh", M, N, K, seed=77)
    _check_full(ora, sp24, w, "heuristic split")


@pytest.mark.parametrize("M,N,K,cs", [(16, 5120, 4096, 2), (1, 5120, 4096, 2), (64, 4096, 4096, 2),
                                      (33, 6144, 2048, 2), (16, 256, 2048, 4), (7, 2560, 4096, 4),
                                      (16, 512, 1024, 2)])
def test_cluster_split(ora, sp24, M, N, K, cs):
    """Cluster split forced: each tile's K range is cut across the cs CTAs of a
    cluster, whose partials reach the leader CTA's shared memory (st.async)
    and are added in rank order; deterministic, and equal to whole tiles
    within rounding."""
    w = inputs.Workload("cl", M, N, K, seed=3 * M + N)
    with sp24.decomposition(sp24.DECOMP_CLUSTER_SPLIT):
        assert sp24.decomposition_of(M, N, K) == (sp24.DECOMP_CLUSTER_SPLIT, cs)
        assert sp24.workspace_size(M, N, K) == 0
        y, ref = _check_full(ora, sp24, w, "cluster split M=%d N=%d K=%d" % (M, N, K))
        xq, sx, values, meta, sw, _, _ = _prep(ora, w)
        y2 = _run_gpu(sp24, w, xq, sx, values, meta, sw, None, None)
    assert np.array_equal(y, y2)


def test_cluster_split_graph_replay(ora, sp24):
    """Cluster-split launches captured in a CUDA graph replay bit-identically."""
    shapes = [(16, 2560, 4096), (64, 1024, 2048)]
    with sp24.decomposition(sp24.DECOMP_CLUSTER_SPLIT):
        cases = []
        for i, (M, N, K) in enumerate(shapes):
            w = inputs.Workload("clg", M, N, K, seed=60 + i)
            xq, sx, values, meta, sw, _, _ = _prep(ora, w)
            tv, tm = _abi(ora, values, meta)
            ops = [dev(t) for t in (xq, sx, tv, tm, sw)]
            y = sp24.gemm(*ops)
            torch.cuda.synchronize()
            sp24.last_device_error()
            assert_close(bf16_to_f64(y), ora.gemm(xq, sx, values, meta, sw), "cluster split shape %d" % i)
            cases.append((ops, y.clone(), torch.empty_like(y)))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for ops, _, out in cases:
                sp24.gemm(*ops, out=out)
    for _ in range(3):
        for _, _, out in cases:
            out.zero_()
        g.replay()
        torch.cuda.synchronize()
        sp24.last_device_error()
        for i, (_, ref, out) in enumerate(cases):
            assert torch.equal(out, ref), "graph replay of shape %d" % i


def test_streamk_workspace_reuse_and_graph_replay(ora, sp24):
    """One workspace, zeroed once, serves calls of different shapes in turn,
    eagerly and as CUDA graph replays: the launch counter's epoch advances on
    the device with every launch, so no flag an earlier launch left is taken
    for a later one's.  Every replay gives the eager result's bits."""
    shapes = [(16, 5120, 4096), (64, 4096, 2048), (7, 2560, 4096)]
    sp24.set_decomposition(sp24.DECOMP_STREAM_K)
    try:
        _reuse_and_replay(ora, sp24, shapes)
    finally:
        sp24.set_decomposition(sp24.DECOMP_HEURISTIC)


def _reuse_and_replay(ora, sp24, shapes):
    ws = torch.zeros(max(sp24.workspace_size(*s) for s in shapes), dtype=torch.uint8, device="cuda")
    cases = []
    for i, (M, N, K) in enumerate(shapes):
        w = inputs.Workload("skr", M, N, K, seed=40 + i)
        xq, sx, values, meta, sw, _, _ = _prep(ora, w)
        tv, tm = _abi(ora, values, meta)
        ops = [dev(t) for t in (xq, sx, tv, tm, sw)]
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        cases.append((ops, y, ora.gemm(xq, sx, values, meta, sw)))
    first = []
    for rep_ in range(2):
        for i, (ops, y, ref) in enumerate(cases):
            sp24.gemm(*ops, out=y, workspace=ws)
            torch.cuda.synchronize()
            sp24.last_device_error()
            if rep_ == 0:
                assert_close(bf16_to_f64(y), ref, "stream-K shape %d" % i)
                first.append(y.clone())
            else:
                assert torch.equal(y, first[i]), "shape %d changed on reuse" % i
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for ops, y, _ in cases:
            sp24.gemm(*ops, out=y, workspace=ws)
    for _ in range(3):
        for _, y, _ in cases:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        sp24.last_device_error()
        for i, (_, y, _) in enumerate(cases):
            assert torch.equal(y, first[i]), "graph replay of shape %d" % i


def test_split_k_without_workspace_runs_unsplit(ora, sp24):
    """A too-small workspace is not an error: the call runs without splitting."""
    M, N, K = 16, 5120, 4096
    w = inputs.Workload("sk0", M, N, K, seed=9)
    xq, sx, values, meta, sw, _, _ = _prep(ora, w)
    tv, tm = _abi(ora, values, meta)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with sp24.decomposition(sp24.DECOMP_STREAM_K):
        y = sp24.gemm(dev(xq), dev(sx), dev(tv), dev(tm), dev(sw), workspace=small)
    torch.cuda.synchronize()
    sp24.last_device_error()
    assert_close(bf16_to_f64(y), ora.gemm(xq, sx, values, meta, sw), "unsplit fallback")


@pytest.mark.parametrize("L,M,N,K,gN,gK,with_bias,mode", [
    (3, 16, 512, 512, 1, None, False, 0),     # decode-size problems: one launch over all of them
    (4, 40, 384, 512, 128, 128, True, 0),     # group-wise promotion, ragged token tails
    (2, 40, 1024, 2048, 1, None, True, 2),    # few tiles: stream-K, each tile cut between 8 CTAs
    (3, 16, 2560, 4096, 1, None, False, 2),   # stream-K ranges that cross tiles and problems
    (3, 16, 2560, 4096, 1, None, True, 3),    # cluster split, one cluster per (problem, tile)
    (3, 300, 512, 512, 1, None, True, 0),     # SM-pair problems: one launch each
    (2, 200, 512, 768, 128, 128, False, 0),   # SM-pair group-wise problems
])
def test_gemm_batched(ora, sp24, L, M, N, K, gN, gK, with_bias, mode):
    """L independent problems of one shape (CUTLASS's batched L mode): each
    output equals the oracle on that problem's own operands.  The activations
    come from a taller buffer, so consecutive problems are not adjacent."""
    gk = K if gK is None else gK
    probs = []
    for l in range(L):
        w = inputs.Workload("batch", M, N, K, gN=gN, gK=gK, seed=100 * l + M + N)
        probs.append((w,) + _prep(ora, w))
    pad = 8
    xq_big = torch.zeros((L, M + pad, K), dtype=torch.uint8)
    for l, p in enumerate(probs):
        xq_big[l, :M] = torch.from_numpy(p[1])
    xq = xq_big.cuda()[:, :M]
    sx = torch.stack([torch.from_numpy(p[2]) for p in probs]).cuda()
    tiled = [_abi(ora, p[3], p[4]) for p in probs]
    values = torch.stack([torch.from_numpy(t[0]) for t in tiled]).cuda()
    meta = torch.stack([torch.from_numpy(t[1]) for t in tiled]).cuda()
    sw = torch.stack([torch.from_numpy(p[5]) for p in probs]).cuda()
    rng = np.random.default_rng(L + M)
    bias_bits = [inputs.bf16_bits(torch.from_numpy(rng.normal(0, 0.5, N).astype(np.float32)).to(torch.bfloat16))
                 for _ in range(L)]
    bias = torch.stack([dev(b) for b in bias_bits]) if with_bias else None
    with sp24.decomposition(mode):
        y = sp24.gemm_batched(xq, sx, values, meta, sw, 1, gN, gk, bias=bias)
    torch.cuda.synchronize()
    sp24.last_device_error()
    for l, p in enumerate(probs):
        ref = ora.gemm(p[1], p[2], p[3], p[4], p[5], 1, gN, gk, bias=bias_bits[l] if with_bias else None)
        assert_close(bf16_to_f64(y[l]), ref, "batched L=%d problem %d" % (L, l))
