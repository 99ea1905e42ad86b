"""Helpers for the GPU parity tests: upload oracle/generator arrays, compare."""
import numpy as np
import torch

RTOL = 1e-2   # |Y - ref| <= RTOL * |ref| + ATOL, element by element
ATOL = 1e-3


def dev(a, dtype=None):
    """numpy array -> CUDA tensor (bit-preserving for uint8/uint16 payloads)."""
    if isinstance(a, torch.Tensor):
        return a.cuda()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(y: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(y - ref)
    bound = RTOL * np.abs(ref) + ATOL
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = ", ".join("(%d,%d): got %.6g ref %.6g" % (i, j, y[i, j], ref[i, j]) for i, j in idx)
        raise AssertionError("%s: %d of %d elements outside %.0e*|ref|+%.0e; first: %s"
                             % (what, int(bad.sum()), bad.size, RTOL, ATOL, msg))
