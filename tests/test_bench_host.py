"""Host-side logic of bench.py, without a GPU: the clock record that decides
whether a timing is kept, the workload descriptions, the table of captured
DRAM traffic (keyed by the full shape, so another shape never borrows a
number), and the peaks file fallback."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import inputs  # noqa: E402


def _sampler(lines):
    c = bench.ClockSampler(0)
    c.lines = list(lines)
    return c.summary()


def test_clock_summary_median_and_reasons():
    lines = [
        "2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1100.5, 0x4, Not Active, Not Active, Not Active, Active",
        "1980, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2055
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_slowdowns():
    lines = ["1500, 2070, 700, 0x8, Active, Not Active, Active, Not Active"] * 3
    s = _sampler(lines)
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples_is_none():
    assert _sampler([]) is None
    assert _sampler(["x, y"]) is None


@pytest.mark.parametrize("name", sorted(bench.DESCR))
def test_descriptions_name_the_shape(name):
    w = inputs.WORKLOADS[name]
    text = bench.DESCR[name].format(N=w.N, K=w.K)
    assert "{" not in text and str(w.K) in text


def test_decode_description_follows_the_shape():
    w = inputs.with_shape(inputs.WORKLOADS["decode"], M=16, N=4096, K=14336)
    text = bench.DESCR["decode"].format(N=w.N, K=w.K)
    assert "W[4096,14336]" in text and "X[M,14336]" in text


def test_captured_traffic_is_keyed_by_the_full_shape():
    """GEMM figures are keyed by (M, N, K), compress figures by (N, K) alone:
    compress reads the weight whatever the token count."""
    for (workload, M, N, K, kernel), traffic in bench.CAPTURED_TRAFFIC.items():
        assert kernel in ("gemm", "compress")
        assert (M is None) == (kernel == "compress")
        w = inputs.WORKLOADS[workload]
        if workload == "decode" and M is not None:
            w = inputs.with_shape(w, M=M)
        assert (w.N, w.K) == (N, K) and M in (None, w.M), "entry for a shape the benchmark does not run"
        assert bench.captured_traffic(workload, w, kernel) == traffic
        for m in inputs.DECODE_M if workload == "decode" and kernel == "compress" else ():
            assert bench.captured_traffic(workload, inputs.with_shape(w, M=m), kernel) == traffic
        # the algorithmic bytes bound the traffic from below (weights read once)
        if kernel == "gemm":
            assert traffic >= N * K * 5 // 8 * 0.95
        else:
            assert traffic >= N * K * 2 * 0.99  # the bf16 weight read once
    other = inputs.with_shape(inputs.WORKLOADS["decode"], M=16, N=4096, K=14336)
    assert bench.captured_traffic("decode", other, "gemm") is None
    assert bench.captured_traffic("decode", other, "compress") is None


def test_peaks_fallback_is_labelled(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6780.7, "bf16_tflops": 1901.0}')
    p = bench.peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 6780.7
    assert p["bf16_tflops_sustained"] == 1901.0


@pytest.mark.parametrize("steps", [1, 3, 5, 7, 50, 51])
def test_replay_split_times_exactly_k_steps(steps):
    split = bench.replay_split(steps)
    assert sum(split) == steps and all(k >= 1 for k in split)
    assert len(split) == min(bench.REPLAYS, steps)
    assert max(split) - min(split) <= 1


def test_default_workload_is_the_largest_single_gpu_config():
    args = bench.parse_args([])
    assert args.workload == "groupwise" and args.multi == "split"
    big = max(inputs.WORKLOADS.values(), key=lambda w: w.dense_flops())
    assert big.name == args.workload


def test_both_arms_describe_the_same_config():
    """The reference arm and the GPU arm print the same config dict: it holds
    only the workload's description, no figure measured at run time."""
    w = inputs.WORKLOADS["groupwise"]
    a = bench.config_dict("groupwise", w, "single")
    assert a == bench.config_dict("groupwise", w, "single")
    assert a["M"] == 3000 and a["N"] == 14336 and a["scales"] == {"gM": 1, "gN": 128, "gK": 128}


def test_algorithmic_counts():
    w = inputs.WORKLOADS["groupwise"]
    assert bench.compress_bytes(w) == w.N * w.K * 21 // 8 + 4 * 32 * 112
    d = inputs.with_shape(inputs.WORKLOADS["decode"], M=16)
    assert bench.gemm_bytes(d) == d.N * d.K * 5 // 8 + 16 * d.K + 2 * 16 * d.N + 4 * (16 + d.N)
    fused = inputs.WORKLOADS["fused"]
    e = bench.tensor_entry(fused, 1.0, 1000.0, 500.0)
    alg, side = fused.dense_flops() / 2, 2.0 * fused.M * fused.N * fused.r
    assert e["frac"] == pytest.approx(round((alg / 1e15 + side / 5e14) / 1e-3, 4))
    assert bench.pair_kernel_applies(w) and bench.pair_kernel_applies(inputs.WORKLOADS["llama"])
    assert not bench.pair_kernel_applies(d)
