"""Benchmark of the 2:4 sparse FP8 hot path on GB300.

One step = one pass of the whole hot path over one batch: compress the bf16
weight (magnitude 2:4 prune + e4m3 + pack) and run the group-wise scaled
sparse GEMM on e4m3 activations.  Activation quantization is input
preparation and runs before the timed region.

The headline workload is the group-wise one (X[3000,4096] with 1x128
activation scales, W[14336,4096] with 128x128 block scales), the largest
configuration that fits one GPU.  Prints ONE JSON line (rank 0).  ``value`` is
dense-equivalent TFLOPS (2*M*N*K per step, the convention sparse tensor peaks
are quoted in) over the whole step, summed over ranks; ``roofline`` describes
the step's dominant kernel.  ``kernels`` carries every configuration's kernels
timed alone (the Llama-style linear, the group-wise GEMM, the decode sweep
and its weight's compression, the fused side GEMM), each against its own
roofline.  ``--impl reference`` times the CPU oracle instead, on a bounded
sample of the same workload.

Timing: CUDA events on the launching stream around CUDA-graph replays (the
kernels run back to back with their programmatic-launch edges, no host gaps),
over rotating input sets larger than L2.  Each figure is the median over
several replays, with the minimum and maximum beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload groupwise]
       torchrun --nproc-per-node N bench.py --gpus N [--multi split|replicas] ...
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import inputs  # noqa: E402

METRIC = "sparse FP8 GEMM TFLOPS & % of FP8 sparse peak; compress GB/s & % HBM peak"
UNIT = "TFLOPS"
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
REPLAYS = 5          # timed graph replays per figure (median, min, max)
# The warp-level int8 sparse MMA's rate on this part (kept-weight TOPS), the
# int8 GEMM's roofline: mma.sp m16n8k64 s8 in a register-only loop.
INT8_MMA_SP_TOPS = 150.6

DESCR = {
    "llama": "Llama-style FP8 linear: X[2048,4096] e4m3 per-token (N(0,1), 0.1% outliers x20), "
             "W[4096,4096] bf16 N(0,0.02) -> 2:4 e4m3 per-channel, Y bf16",
    "groupwise": "group-wise scaling: X[3000,4096] e4m3 with 1x128 activation scales (partial M tile), "
                 "W[14336,4096] bf16 N(0,0.02) -> 2:4 e4m3 with 128x128 block scales, Y bf16",
    "fused": "fused: llama shapes + bf16 side GEMM X2[2048,64] W2[4096,64]",
    "decode": "decode: X[M,{K}] per-token, W[{N},{K}] per-channel",
    "tiny": "tiny: X[128,512], W[256,512]",
}


# DRAM bytes (read + write) per launch of a kernel, from one ncu capture of
# the current kernel build (summaries and commands under profiles/).  An entry
# is removed when its kernel changes; absent entries report null.
CAPTURED_TRAFFIC = {
    # sp24_gemm_pair_kernel<240,0,0> on the Llama-style linear (M 2048, N 4096, K 4096)
    ("llama", 2048, 4096, 4096, "gemm"): 18939648 + 0,
    # sp24_gemm_kernel<16,0,0,0,4,0> (whole tiles), decode M 16, N 28672, K 4096
    ("decode", 16, 28672, 4096, "gemm"): 73608192 + 411392,
    # sp24_gemm_pair_kernel<240,1,0>, fused side GEMM M 2048, N 4096, K 4096, r 64
    ("fused", 2048, 4096, 4096, "gemm"): 19725312 + 0,
    # sp24_gemm_pair_kernel<128,0,1>, group-wise M 3000, N 14336, K 4096
    ("groupwise", 3000, 14336, 4096, "gemm"): 51097088 + 55554048,
    # compress (no token count): compress_rows_pipe_kernel<8>, W 4096 x 4096 (the
    # output stays in L2)
    ("llama", None, 4096, 4096, "compress"): 33623296 + 256,
    # compress_rows_pipe_kernel<8>, W 28672 x 4096
    ("decode", None, 28672, 4096, "compress"): 234967808 + 17726976,
    # compress_blocks_kernel, W 14336 x 4096, 128 x 128 block scales
    ("groupwise", None, 14336, 4096, "compress"): 117484800 + 6699520,
}


def compress_kernel(w):
    """The kernel sp24_fp8_compress runs for this workload's weight."""
    if w.gN == 128:
        return "compress_blocks_kernel"
    return "compress_rows_pipe_kernel" if w.gk == w.K and w.K <= 4096 else "compress_rows_kernel"


def captured_traffic(workload, w, kernel):
    return CAPTURED_TRAFFIC.get((workload, None if kernel == "compress" else w.M, w.N, w.K, kernel))


# ------------------------------------------------------ algorithmic counts
def n_scales(K, gk, rows, g):
    return (K // gk) * ((rows + g - 1) // g)


def compress_bytes(w):
    """W read once + kept values, metadata and scales written (2.625 B per weight)."""
    return w.N * w.K * 2 + w.N * w.K // 2 + w.N * w.K // 8 + 4 * n_scales(w.K, w.gk, w.N, w.gN)


def gemm_bytes(w):
    """Operands read once + Y written: values, metadata, activations, scales, side operands."""
    side = 2 * w.r * (w.M + w.N)
    return (w.N * w.K // 2 + w.N * w.K // 8 + w.M * w.K + 2 * w.M * w.N + side
            + 4 * (n_scales(w.K, w.gk, w.M, w.gM) + n_scales(w.K, w.gk, w.N, w.gN)))


def pair_kernel_applies(w):
    """The library's SM-pair rules: plain scaling above 192 tokens (side rank
    at most 64), group-wise above 64 tokens with whole two-block stages."""
    if w.N % 256 != 0:
        return False
    if w.gk == w.K:
        return w.r <= 64 and w.M > 192
    return w.gk == 128 and w.K > 128 and w.r == 0 and w.M > 64 and (w.K // 128) % 2 == 0


def spread(ms_list, per=1):
    """Median, min and max of per-launch times (ms) from a list of replay times."""
    v = sorted(x / per for x in ms_list)
    return {"ms": round(statistics.median(v), 5), "ms_min": round(v[0], 5), "ms_max": round(v[-1], 5),
            "replays": len(v)}


def tensor_entry(w, t, peak_fp8_dense, peak_bf16):
    """Roofline of a tensor-bound GEMM: algorithmic flops (kept weights only)
    against the fp8 dense peak, plus the side GEMM's bf16 flops against the
    bf16 peak (the combined roofline time of the fused kernel)."""
    alg = w.dense_flops() / 2
    side = 2.0 * w.M * w.N * w.r
    t_roof = alg / (peak_fp8_dense * 1e12) + side / (peak_bf16 * 1e12)
    return {"bound": "tensor", "achieved": round((alg + side) / (t * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "tflops_dense_equiv": round(w.dense_flops() / (t * 1e-3) / 1e12, 1),
            "frac": round(t_roof / (t * 1e-3), 4)}


def hbm_entry(nbytes, t, peak_hbm):
    gbs = nbytes / (t * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak_hbm, 4),
            "bytes": int(nbytes)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(w, world, rank, multi):
    """This rank's share of the workload.  split: the weight rows of
    shard.shard_rows (whole 128-row tiles) with the full activations, a
    disjoint block of Y's columns and no exchange; replicas: the whole
    layer on a batch of its own."""
    if world == 1:
        return w, (0, w.N)
    if multi == "split":
        from semi_structured_sparse_gb300 import shard
        a, b = shard.shard_rows(w.N, world, rank)
        return inputs.with_shape(w, N=b - a), (a, b)
    return inputs.with_shape(w, seed=w.seed + 1000 * rank), (0, w.N)


# ------------------------------------------------------------- our GPU arm
class Bench:
    """Device-resident rotating input sets of one workload and graph timing."""

    def __init__(self, sp24, w, dev, stream, X=None, W=None, X2=None, W2=None, weights_from=None):
        self.sp24, self.w, self.dev, self.stream = sp24, w, dev, stream
        if X is None:
            X, W, X2, W2 = inputs.generate(w)
        self.X, self.W, self.X2, self.W2 = X, W, X2, W2
        gk = w.gk
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.set_bytes = (w.N * w.K * 2 + w.M * w.K + w.N * w.K // 2 + w.N * w.K // 8 + w.M * w.N * 2)
        gemm_operands = w.N * w.K // 2 + w.N * w.K // 8 + w.M * w.K
        if weights_from is not None:
            # decode token counts share the weight sets of one workload: only the
            # activations and outputs are per set
            self.nsets = weights_from.nsets
        else:
            # enough sets that both the compress inputs and the GEMM operands
            # of the other sets exceed 3x L2 between two uses of a set
            self.nsets = max(2, -(-3 * l2 // self.set_bytes), -(-3 * l2 // gemm_operands))
        self.l2 = l2
        self.xq0, self.sx0 = sp24.quantize_act(X.to(dev), gk)
        Wd = None if weights_from is not None else W.to(dev)
        self.sets = []
        for i in range(self.nsets):
            if weights_from is not None:
                src = weights_from.sets[i]
                s = {k: src[k] for k in ("W", "v", "m", "sw")}
            else:
                s = {"W": Wd.clone(),
                     "v": torch.empty((w.N, w.K // 2), dtype=torch.uint8, device=dev),
                     "m": torch.empty((w.N, w.K // 8), dtype=torch.uint8, device=dev),
                     "sw": torch.empty((w.K // gk, (w.N + w.gN - 1) // w.gN), dtype=torch.float32, device=dev)}
            s.update({"xq": self.xq0.clone(), "sx": self.sx0.clone(),
                      "y": torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev),
                      "x2": None if X2 is None else X2.to(dev), "w2": None if W2 is None else W2.to(dev)})
            self.sets.append(s)
        self.ws_bytes = sp24.workspace_size(w.M, w.N, w.K, w.r)
        self.ws = torch.zeros(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        if weights_from is None:
            for s in self.sets:
                self.compress(s)
        torch.cuda.synchronize()

    def compress(self, s):
        w = self.w
        self.sp24.compress(s["W"], w.gN, w.gk, out=(s["v"], s["m"], s["sw"]))

    def gemm(self, s):
        w = self.w
        self.sp24.gemm(s["xq"], s["sx"], s["v"], s["m"], s["sw"], w.gM, w.gN, w.gk, s["x2"], s["w2"],
                       out=s["y"], workspace=self.ws)

    def step(self, s):
        self.compress(s)
        self.gemm(s)

    def capture(self, fn, n, offset=0):
        """A CUDA graph of n calls fn(set) over the rotating sets: replayed, the
        kernels run back to back with their programmatic-launch edges."""
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(self.dev)
        cs.wait_stream(self.stream)
        with torch.cuda.stream(cs):
            with torch.cuda.graph(g, stream=cs):
                for i in range(n):
                    fn(self.sets[(offset + i) % self.nsets])
        self.stream.wait_stream(cs)
        torch.cuda.synchronize()
        return g

    def time_replays(self, g, reps):
        """Replay g reps times, one event pair per replay on the launching stream."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        g.replay()  # warm, untimed
        torch.cuda.synchronize()
        ev[0].record(self.stream)
        for i in range(reps):
            g.replay()
            ev[i + 1].record(self.stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]

    def time_kernel(self, fn, n, reps=REPLAYS):
        for i in range(3):
            fn(self.sets[i % self.nsets])
        torch.cuda.synchronize()
        g = self.capture(fn, n)
        r = self.time_replays(g, reps)
        self.sp24.last_device_error()
        return spread(r, n)


def gemm_schedule(sp24, w, ws_bytes):
    if pair_kernel_applies(w):
        return "sp24_gemm_pair_kernel", "whole tiles"
    if w.gk != w.K or w.r:
        return "sp24_gemm_kernel", "whole tiles"
    mode, cs = sp24.decomposition_of(w.M, w.N, w.K, w.r)
    sched = {sp24.DECOMP_STREAM_K: "stream-K" if ws_bytes else "whole tiles",
             sp24.DECOMP_CLUSTER_SPLIT: "cluster split-K, %d CTAs per tile" % cs}.get(mode, "whole tiles")
    return "sp24_gemm_kernel", sched


def other_configs(sp24, dev, stream, headline, pk, n):
    """Every configuration's kernels, each alone (a graph of n launches over
    rotating sets larger than L2, replayed REPLAYS times): the Llama-style
    linear (GEMM, compress), the fused side GEMM, the decode sweep (GEMM at
    every token count, compress of its weight), plus the headline workload's
    own kernels, which the caller adds."""
    fp8 = pk["bf16_tflops"] * FP8_OVER_BF16
    out = {}

    def gemm_row(name, b, wl):
        t = b.time_kernel(b.gemm, n)
        kern, sched = gemm_schedule(sp24, b.w, b.ws_bytes)
        row = dict(t, kernel=kern, schedule=sched, M=b.w.M, N=b.w.N, K=b.w.K)
        if b.w.M > 64:
            row.update(tensor_entry(b.w, t["ms"], fp8, pk["bf16_tflops"]))
        else:
            row.update(hbm_entry(gemm_bytes(b.w), t["ms"], pk["hbm_gbs"]))
        row["traffic"] = captured_traffic(wl, b.w, "gemm")
        out[name] = row

    def compress_row(name, b, wl):
        t = b.time_kernel(b.compress, n)
        kern = compress_kernel(b.w)
        out[name] = dict(t, kernel=kern, N=b.w.N, K=b.w.K, traffic=captured_traffic(wl, b.w, "compress"),
                         **hbm_entry(compress_bytes(b.w), t["ms"], pk["hbm_gbs"]))

    for wl in ("llama", "fused"):
        if wl == headline:
            continue
        b = Bench(sp24, inputs.WORKLOADS[wl], dev, stream)
        gemm_row(wl + "_gemm", b, wl)
        if wl == "llama":
            compress_row("llama_compress", b, wl)
            out.update(int8_rows(sp24, b, pk, n))
        del b
    if headline != "groupwise":
        b = Bench(sp24, inputs.WORKLOADS["groupwise"], dev, stream)
        gemm_row("groupwise_gemm", b, "groupwise")
        compress_row("groupwise_compress", b, "groupwise")
        del b
    base = None
    for M in inputs.DECODE_M:
        wd = inputs.with_shape(inputs.WORKLOADS["decode"], M=M)
        if base is None:
            base = Bench(sp24, wd, dev, stream)
            compress_row("decode_compress", base, "decode")
            b = base
        else:
            X, _, _, _ = inputs.generate(wd) if M != base.w.M else (base.X, None, None, None)
            b = Bench(sp24, wd, dev, stream, X=X, W=base.W, weights_from=base)
        gemm_row("decode_gemm_M%d" % M, b, "decode")
    torch.cuda.synchronize()
    return out


def int8_rows(sp24, b, pk, n):
    """The int8 x int8 2:4 sibling on the Llama-style linear's shape and
    rotating sets (per-token x per-channel int8): its compress (HBM-bound) and
    its GEMM, which runs on the warp-level sparse MMA (sm_103a has no int8
    tcgen05 MMA).  The GEMM's peak is that instruction's own rate on this part,
    measured with a register-only loop of it: 150.6 TOPS of kept-weight work
    (0.062 MMA per clock per SM at 4 to 16 warps per SM)."""
    w = b.w
    for s in b.sets:
        s["v8"], s["m8"], s["sw8"] = sp24.compress_int8(s["W"])
        s["xq8"], s["sx8"] = sp24.quantize_act_int8(b.X.to(b.dev))
    torch.cuda.synchronize()
    t_g = b.time_kernel(lambda s: sp24.gemm_int8(s["xq8"], s["sx8"], s["v8"], s["m8"], s["sw8"], out=s["y"]), n)
    t_c = b.time_kernel(lambda s: sp24.compress_int8(s["W"], out=(s["v8"], s["m8"], s["sw8"])), n)
    ops = w.M * w.N * w.K  # 2 M N K / 2: kept weights only
    fp8 = pk["bf16_tflops"] * FP8_OVER_BF16
    achieved = ops / (t_g["ms"] * 1e-3) / 1e12
    c_bytes = w.N * w.K * 2 + w.N * w.K // 2 + w.N * w.K // 8 + 4 * w.N
    for s in b.sets:
        for k in ("v8", "m8", "sw8", "xq8", "sx8"):
            del s[k]
    return {
        "llama_int8_gemm": dict(t_g, kernel="sp24_int8_gemm_kernel", M=w.M, N=w.N, K=w.K, bound="tensor",
                                achieved=round(achieved, 1), unit="TOPS", peak=INT8_MMA_SP_TOPS,
                                frac=round(achieved / INT8_MMA_SP_TOPS, 4),
                                peak_source="mma.sp m16n8k64 s8 in a register-only loop on this part",
                                frac_of_fp8_peak=round(achieved / fp8, 4),
                                counts="2*M*N*K/2 int8 operations (kept weights only)"),
        "llama_int8_compress": dict(t_c, kernel=compress_kernel(w) + " (int8 codes)",
                                    N=w.N, K=w.K, **hbm_entry(c_bytes, t_c["ms"], pk["hbm_gbs"])),
    }


def next_rows(sp24, b, pk, n):
    """The §8(f) kernels on the headline workload, each alone: the GEMM with a
    bf16 bias, a batch of 4 problems, activation quantization from bf16, and
    the GPU dequantize."""
    w, sets, gk = b.w, b.sets, b.w.gk
    dev = sets[0]["y"].device
    bias = [torch.randn(w.N, device=dev).to(torch.bfloat16) for _ in sets]
    xb = [torch.randn(w.M, w.K, device=dev).to(torch.bfloat16) for _ in sets]
    qx = [(torch.empty_like(s["xq"]), torch.empty_like(s["sx"])) for s in sets]
    dq = [torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev) for _ in sets]
    idx = {id(s): i for i, s in enumerate(sets)}

    def gemm_bias(s):
        sp24.gemm(s["xq"], s["sx"], s["v"], s["m"], s["sw"], w.gM, w.gN, gk, s["x2"], s["w2"], out=s["y"],
                  workspace=b.ws, bias=bias[idx[id(s)]])

    t_bias = b.time_kernel(gemm_bias, n)
    L = 4
    s0 = sets[0]
    bx = s0["xq"].unsqueeze(0).repeat(L, 1, 1)
    bsx = s0["sx"].unsqueeze(0).repeat(L, 1, 1)
    bv = s0["v"].unsqueeze(0).repeat(L, 1, 1)
    bm = s0["m"].unsqueeze(0).repeat(L, 1, 1)
    bsw = s0["sw"].unsqueeze(0).repeat(L, 1, 1)
    by = torch.empty((L, w.M, w.N), dtype=torch.bfloat16, device=dev)
    bws = torch.zeros(max(16, L * sp24.workspace_size(w.M, w.N, w.K)), dtype=torch.uint8, device=dev)
    t_batch = b.time_kernel(lambda s: sp24.gemm_batched(bx, bsx, bv, bm, bsw, w.gM, w.gN, gk, out=by,
                                                        workspace=bws), max(3, n // 4))
    t_q = b.time_kernel(lambda s: sp24.quantize_act(xb[idx[id(s)]], gk, out=qx[idx[id(s)]]), n)
    t_d = b.time_kernel(lambda s: sp24.decompress(s["v"], s["m"], s["sw"], w.gN, gk, out=dq[idx[id(s)]]), n)
    q_bytes = w.M * w.K * 2 + w.M * w.K + 4 * n_scales(w.K, gk, w.M, 1)
    d_bytes = w.N * w.K // 2 + w.N * w.K // 8 + 4 * n_scales(w.K, gk, w.N, w.gN) + 2 * w.N * w.K
    fp8 = pk["bf16_tflops"] * FP8_OVER_BF16
    return {
        "gemm_with_bias": dict(t_bias, **tensor_entry(w, t_bias["ms"], fp8, pk["bf16_tflops"])),
        "gemm_batched": dict(t_batch, L=L, **tensor_entry(inputs.with_shape(w, M=L * w.M), t_batch["ms"], fp8,
                                                             pk["bf16_tflops"])),
        "quantize_act_bf16": dict(t_q, **hbm_entry(q_bytes, t_q["ms"], pk["hbm_gbs"]),
                                  counts="M*K*2 read + M*K + scales written"),
        "decompress": dict(t_d, **hbm_entry(d_bytes, t_d["ms"], pk["hbm_gbs"]),
                           counts="N*K/2 values + N*K/8 metadata + scales read, N*K*2 written"),
    }


def e2e_pass(sp24, b, steps, warm, pg):
    """End to end through the public API with host buffers: every step uploads
    its inputs from pinned host memory and downloads its output.  Two buffer
    sets and two copy streams let step i + 1's upload and step i - 1's
    download overlap step i's kernels; each step still moves all its bytes."""
    w, dev, stream = b.w, b.dev, b.stream
    pin_W = b.W.pin_memory()
    pin_xq = b.xq0.cpu().pin_memory()
    pin_sx = b.sx0.cpu().pin_memory()
    pin_x2 = None if b.X2 is None else b.X2.pin_memory()
    pin_w2 = None if b.W2 is None else b.W2.pin_memory()
    pin_y = [torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    bufs = b.sets[:2]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set i uploaded
    ev_done = [torch.cuda.Event() for _ in range(2)]  # kernels on set i finished (inputs free, output ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # output of set i downloaded
    used = [False, False]

    def one(i):
        k = i % 2
        s = bufs[k]
        with torch.cuda.stream(up):
            if used[k]:
                up.wait_event(ev_done[k])  # the previous step on this set has read its inputs
            s["W"].copy_(pin_W, non_blocking=True)
            s["xq"].copy_(pin_xq, non_blocking=True)
            s["sx"].copy_(pin_sx, non_blocking=True)
            if pin_x2 is not None:
                s["x2"].copy_(pin_x2, non_blocking=True)
                s["w2"].copy_(pin_w2, non_blocking=True)
            ev_in[k].record(up)
        stream.wait_event(ev_in[k])
        if used[k]:
            stream.wait_event(ev_out[k])  # this set's previous output has been downloaded
        b.step(s)
        ev_done[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[k])
            pin_y[k].copy_(s["y"], non_blocking=True)
            ev_out[k].record(down)
        used[k] = True

    i = 0
    for _ in range(warm):
        one(i)
        i += 1
    torch.cuda.synchronize()
    # the median of REPLAYS timed runs of `steps` steps each, so that one run
    # slowed by other traffic on the host link does not set the figure
    runs = []
    for _ in range(REPLAYS):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if pg:
            pg.barrier()
        e0.record(stream)
        up.wait_stream(stream)
        for _ in range(steps):
            one(i)
            i += 1
        stream.wait_stream(down)
        e1.record(stream)
        torch.cuda.synchronize()
        runs.append(e0.elapsed_time(e1) / steps)
    ms = sorted(runs)[len(runs) // 2]
    h2d = (pin_W.numel() * 2 + pin_xq.numel() + pin_sx.numel() * 4
           + (0 if pin_x2 is None else pin_x2.numel() * 2 + pin_w2.numel() * 2))
    return ms, int(h2d), int(pin_y[0].numel() * 2)


def replay_split(steps):
    """Steps per timed replay: REPLAYS replays (fewer if K is smaller) whose
    step counts add up to exactly K."""
    r = max(1, min(REPLAYS, steps))
    q, extra = divmod(steps, r)
    return [q + (1 if i < extra else 0) for i in range(r)]


def run_ours(args):
    import semi_structured_sparse_gb300 as sp24

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    sp24.load(build_if_missing=(world == 1))
    w0 = inputs.WORKLOADS[args.workload]
    if args.workload == "decode":
        w0 = inputs.with_shape(w0, M=args.decode_m, N=args.decode_n, K=args.decode_k)
    w, rows = rank_workload(w0, world, rank, args.multi)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if world > 1 and args.multi == "split":
        # this rank's rows of the one layer's weight, with the full activations
        X, W, X2, W2 = inputs.generate(w0)
        a, e = rows
        b = Bench(sp24, w, dev, stream, X=X, W=W[a:e].contiguous(), X2=X2,
                  W2=None if W2 is None else W2[a:e].contiguous())
    else:
        b = Bench(sp24, w, dev, stream)

    for i in range(args.warmup):
        b.step(b.sets[i % b.nsets])
    torch.cuda.synchronize()
    sp24.last_device_error()

    # the timed steps: exactly K whole steps, cut into replays of graphs whose
    # step counts add up to K (one event pair per replay)
    split = replay_split(args.steps)
    graphs, off = [], 0
    for k in split:
        graphs.append(b.capture(b.step, k, offset=off))
        off += k
    n_k = max(args.steps, 3)
    g_comp = b.capture(b.compress, n_k)
    g_gemm = b.capture(b.gemm, n_k)
    for g in graphs + [g_comp, g_gemm]:  # warm replays, untimed
        g.replay()
    torch.cuda.synchronize()
    sp24.last_device_error()

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
    with ClockSampler(local) as clk:
        # keep the GPU busy ~1 s so the clock samples see it under load, untimed
        t_end = time.time() + (0.0 if args.quick else 1.0)
        i = 0
        while time.time() < t_end:
            graphs[0].replay()
            i += 1
            if i % 4 == 0:
                torch.cuda.synchronize()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for j, g in enumerate(graphs):
            g.replay()
            ev[j + 1].record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        # each kernel alone for the roofline: a graph of launches over the
        # same rotating sets, replayed REPLAYS times between event pairs
        t_comp = spread(b.time_replays(g_comp, REPLAYS), n_k)
        t_gemm = spread(b.time_replays(g_gemm, REPLAYS), n_k)
    sp24.last_device_error()
    per_step = sorted(ev[j].elapsed_time(ev[j + 1]) / k for j, k in enumerate(split))
    total_ms = sum(ev[j].elapsed_time(ev[j + 1]) for j in range(len(split)))
    ms_step = statistics.median(per_step)
    if pg:
        t = torch.tensor([ms_step, total_ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms_step, total_ms = float(t[0].item()), float(t[1].item())

    e2e_ms, h2d, d2h = (None, 0, 0)
    if not args.quick:
        e2e_ms, h2d, d2h = e2e_pass(sp24, b, max(3, min(args.steps, 20)), max(3, args.warmup), pg)
        if pg:
            t = torch.tensor([e2e_ms], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            e2e_ms = float(t.item())

    pk = peaks()
    fp8 = pk["bf16_tflops"] * FP8_OVER_BF16
    # units of work: the whole layer's flops when the ranks split it, each
    # replica's own batch otherwise
    job_flops = w0.dense_flops() if (world > 1 and args.multi == "split") else world * w.dense_flops()
    kern, sched = gemm_schedule(sp24, w, b.ws_bytes)
    gemm_row = dict(t_gemm, kernel=kern, schedule=sched, M=w.M, N=w.N, K=w.K,
                    traffic=captured_traffic(args.workload, w, "gemm"),
                    **(tensor_entry(w, t_gemm["ms"], fp8, pk["bf16_tflops"]) if w.M > 64
                       else hbm_entry(gemm_bytes(w), t_gemm["ms"], pk["hbm_gbs"])))
    comp_kernel = compress_kernel(w)
    comp_row = dict(t_comp, kernel=comp_kernel, N=w.N, K=w.K, traffic=captured_traffic(args.workload, w, "compress"),
                    **hbm_entry(compress_bytes(w), t_comp["ms"], pk["hbm_gbs"]))
    kernels = {args.workload + "_gemm": gemm_row, args.workload + "_compress": comp_row}
    extra = None
    if world == 1 and not args.quick:
        kernels.update(other_configs(sp24, dev, stream, args.workload, pk, n_k))
        extra = next_rows(sp24, b, pk, n_k)
        for k in [k for k in kernels if "_int8_" in k]:  # the int8 sibling is a next row, not a configuration
            extra[k] = kernels.pop(k)
    # the dominant kernel of the step
    if t_gemm["ms"] >= t_comp["ms"]:
        g = gemm_row
        if g["bound"] == "tensor":
            roofline = {"kernel": g["kernel"], "bound": "tensor", "achieved": g["achieved"], "peak": round(fp8, 1),
                        "unit": "TFLOP/s", "frac": g["frac"], "traffic": g["traffic"],
                        "peak_source": "%s bf16 burst x %.0f (nominal fp8/bf16), of %s" % (
                            pk["source"], FP8_OVER_BF16, pk["source"]),
                        "achieved_counts": "algorithmic 2*M*N*K/2 flops (kept weights only) per launch",
                        "ms": g["ms"]}
        else:
            roofline = {"kernel": g["kernel"], "bound": "hbm", "achieved": g["achieved"],
                        "peak": round(pk["hbm_gbs"], 1), "unit": "GB/s", "frac": g["frac"], "traffic": g["traffic"],
                        "peak_source": "%s copy bandwidth, of %s" % (pk["source"], pk["source"]),
                        "achieved_counts": "algorithmic bytes per launch: operands read once, Y written",
                        "ms": g["ms"]}
    else:
        roofline = {"kernel": comp_kernel, "bound": "hbm", "achieved": comp_row["achieved"],
                    "peak": round(pk["hbm_gbs"], 1), "unit": "GB/s", "frac": comp_row["frac"],
                    "traffic": comp_row["traffic"],
                    "peak_source": "%s copy bandwidth, of %s" % (pk["source"], pk["source"]),
                    "achieved_counts": "algorithmic bytes per launch: W read + values, metadata, scales written",
                    "ms": comp_row["ms"]}
    mode = "single" if world == 1 else ("split along N, %d rows on rank 0" % (rows[1] - rows[0])
                                        if args.multi == "split" else "replicas")
    out = {
        "metric": METRIC,
        "value": round(job_flops / (ms_step * 1e-3) / 1e12, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "ms_per_step_spread": {"min": round(per_step[0], 5), "max": round(per_step[-1], 5),
                               "mean": round(total_ms / args.steps, 5), "replays": len(split)},
        "higher_is_better": True,
        "scaling": "strong" if (world > 1 and args.multi == "split") else "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": config_dict(args.workload, w0, mode),
        "input_sets": {"sets": b.nsets, "mb_per_set": round(b.set_bytes / 1e6, 1), "l2_mb": round(b.l2 / 1e6, 1)},
        "kernels": kernels,
        "roofline": roofline,
        "e2e": None if e2e_ms is None else {
            "value": round(job_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "pipelining": "two buffer sets; step i+1's upload and step i-1's download overlap step i"},
        "next_rows": extra,
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not (args.no_cpu_baseline or args.quick):
        out["cpu_baseline"] = cpu_baseline(w0, budget_s=args.cpu_budget)
    if pg:
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def config_dict(workload, w, parallelism):
    """The workload and timing description, the same in both arms."""
    l2_text = ("inputs larger than L2: rotating input sets, the GEMM operands and the compress inputs "
               "of the other sets each exceed 3x L2 between two uses of a set")
    return {"workload": DESCR[workload].format(N=w.N, K=w.K), "M": w.M, "N": w.N, "K": w.K,
            "scales": {"gM": w.gM, "gN": w.gN, "gK": w.gk}, "side_r": w.r,
            "step": "compress(W) + sparse GEMM", "flops_per_step": "2*M*N*K dense-equivalent",
            "l2": l2_text, "parallelism": parallelism,
            "timing": "value: exactly K steps, as %d CUDA-graph replays between event pairs, median per-step "
                      "time; kernels/roofline: each kernel alone, a graph of launches over the same rotating "
                      "sets, median of %d replays; e2e: eager calls through the public API, median of %d timed runs"
                      % (REPLAYS, REPLAYS, REPLAYS)}


# ------------------------------------------------------------ oracle (CPU)
def cpu_step_estimate(w: inputs.Workload, budget_s: float):
    """Time the oracle on a bounded sample of the workload and scale it to one
    whole step (compress all of W + GEMM of all M tokens).
    Returns (seconds per step, description, threads)."""
    import oracle
    X, W, X2, W2 = inputs.generate(w)
    gk = w.gk
    Wb = inputs.bf16_bits(W)
    # compress sample: whole 128-row blocks
    n_rows = min(w.N, 512)
    t0 = time.perf_counter()
    values, meta, sw = oracle.compress(Wb[:n_rows], w.gN, gk)
    t_comp = (time.perf_counter() - t0) * (w.N / n_rows)
    values, meta, sw = oracle.compress(Wb, w.gN, gk)
    xq, sx = oracle.quantize_act(X.numpy(), gk)
    # GEMM sample: the first m_s tokens, sized to the time budget
    m_s = 1
    t_g = 0.0
    while True:
        t0 = time.perf_counter()
        oracle.gemm(xq[:m_s], sx[:, :m_s], values, meta, sw, 1, w.gN, gk,
                    None if X2 is None else inputs.bf16_bits(X2)[:m_s], None if W2 is None else inputs.bf16_bits(W2))
        t_g = time.perf_counter() - t0
        if t_g > budget_s / 8 or m_s >= w.M:
            break
        m_s = min(w.M, m_s * 4)
    t_gemm = t_g * (w.M / m_s)
    descr = ("oracle compress of %d of %d weight rows and GEMM of %d of %d token rows (all N, K), "
             "scaled to the full step" % (n_rows, w.N, m_s, w.M))
    return t_comp + t_gemm, descr, oracle.num_threads()


def cpu_baseline(w, budget_s=20.0):
    sec, descr, threads = cpu_step_estimate(w, budget_s)
    return {"value": round(w.dense_flops() / sec / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": descr, "seconds_per_step": round(sec, 3)}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return  # the CPU reference arm runs on rank 0 only
    w = inputs.WORKLOADS[args.workload]
    if args.workload == "decode":
        w = inputs.with_shape(w, M=args.decode_m, N=args.decode_n, K=args.decode_k)
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    secs = []
    descr, threads = "", 1
    for i in range(args.warmup + args.steps):
        s, descr, threads = cpu_step_estimate(w, budget)
        if i >= args.warmup:
            secs.append(s)
    sec = statistics.median(secs)
    value = w.dense_flops() / sec / 1e12
    out = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
        "scaling": "strong" if (world > 1 and args.multi == "split") else "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic", "impl": "reference",
        "config": config_dict(args.workload, w, "single" if world == 1 else (
            "split along N" if args.multi == "split" else "replicas")),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": descr},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(inputs.WORKLOADS), default="groupwise")
    ap.add_argument("--multi", choices=["split", "replicas"], default="split",
                    help="N > 1: split the weight rows across ranks (no exchange), or run replicas")
    ap.add_argument("--decode-m", type=int, default=16)
    ap.add_argument("--decode-n", type=int, default=None,
                    help="decode workload: another weight height (default 28672)")
    ap.add_argument("--decode-k", type=int, default=None,
                    help="decode workload: another K (default 4096)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no clock soak, no e2e pass, no other configs, no CPU baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    return args


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
