"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random tensors (and rounds them to the storage type the
workload names); it contains none of the method's arithmetic -- no pruning, no
scaling, no quantization.  Both the oracle and the CUDA path consume the same
bytes produced here.

Workloads (token count M, output channels N, reduction K):

* ``tiny``       -- M128 N256 K512, per-token x per-channel scales, seed 0;
* ``llama``      -- M2048 N4096 K4096, activations N(0,1) with 0.1 % outliers x20;
* ``groupwise``  -- M3000 N14336 K4096, 1x128 activation / 128x128 weight scales;
* ``decode``     -- M in {1,8,16,32,64}, N28672 K4096 (plus compress of that W);
* ``fused``      -- as ``llama`` plus a bf16 rank-64 side GEMM X2[2048,64] W2[4096,64].

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; tensors drawn in the
order X, W, outlier positions, X2, W2; W = bf16(0.02 * N(0,1)); X = N(0,1) in
fp32; outliers: round(frac * M * K) distinct positions chosen uniformly and
multiplied by 20 before quantization; X2 = bf16(N(0,1)); W2 = bf16(0.02 * N(0,1)).
"""
from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    gM: int = 1          # activation scale rows per group (1 = per token)
    gN: int = 1          # weight scale rows per group (1 = per channel)
    gK: Optional[int] = None  # scale K block (None = K, one block)
    outlier_frac: float = 0.0
    outlier_mult: float = 20.0
    r: int = 0           # side-GEMM rank (0 = none)
    seed: int = 0

    @property
    def gk(self) -> int:
        return self.K if self.gK is None else self.gK

    def dense_flops(self) -> float:
        """2*M*N*K: the dense-equivalent count in which sparse peaks are quoted."""
        return 2.0 * self.M * self.N * self.K


WORKLOADS = {
    "tiny": Workload("tiny", 128, 256, 512, seed=0),
    "llama": Workload("llama", 2048, 4096, 4096, outlier_frac=0.001, seed=1),
    "groupwise": Workload("groupwise", 3000, 14336, 4096, gM=1, gN=128, gK=128, seed=2),
    "decode": Workload("decode", 1, 28672, 4096, seed=3),
    "fused": Workload("fused", 2048, 4096, 4096, r=64, seed=4),
}

DECODE_M = (1, 8, 16, 32, 64)


def with_shape(w: Workload, M: Optional[int] = None, N: Optional[int] = None,
               K: Optional[int] = None, seed: Optional[int] = None) -> Workload:
    """Same scale structure and value distribution at another size."""
    kw = {}
    if M is not None:
        kw["M"] = M
    if N is not None:
        kw["N"] = N
    if K is not None:
        kw["K"] = K
    if seed is not None:
        kw["seed"] = seed
    return replace(w, **kw)


def generate(w: Workload):
    """Draw (X fp32 [M,K], W bf16 [N,K], X2 bf16 [M,r] | None, W2 bf16 [N,r] | None)."""
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    X = torch.randn((w.M, w.K), generator=g, dtype=torch.float32)
    W = (0.02 * torch.randn((w.N, w.K), generator=g, dtype=torch.float32)).to(torch.bfloat16)
    if w.outlier_frac > 0:
        n_out = int(round(w.outlier_frac * w.M * w.K))
        pos = torch.randperm(w.M * w.K, generator=g)[:n_out]
        flat = X.view(-1)
        flat[pos] = flat[pos] * w.outlier_mult
    X2 = W2 = None
    if w.r > 0:
        X2 = torch.randn((w.M, w.r), generator=g, dtype=torch.float32).to(torch.bfloat16)
        W2 = (0.02 * torch.randn((w.N, w.r), generator=g, dtype=torch.float32)).to(torch.bfloat16)
    return X, W, X2, W2


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
