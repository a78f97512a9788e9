"""Helpers for the GPU parity tests: guarded device buffers and the
comparison metrics the tolerances are stated in."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

GUARD = 4096  # bytes of canary on each side of a guarded buffer
CANARY = 0xA5


class Guarded:
    """A device buffer of n elements with canary bytes before and after it.
    ``view`` is 16-byte aligned; ``intact()`` checks the canaries."""

    def __init__(self, n: int, dtype: torch.dtype, device: str = "cuda"):
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = n * esize
        self.base = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.view = self.base[GUARD:GUARD + self.nbytes].view(dtype)
        assert self.view.data_ptr() % 16 == 0

    def intact(self) -> bool:
        head = self.base[:GUARD]
        tail = self.base[GUARD + self.nbytes:]
        return bool(torch.all(head == CANARY)) and bool(torch.all(tail == CANARY))


def to_dev_bf16(a: np.ndarray, out: torch.Tensor | None = None) -> torch.Tensor:
    """uint16 bf16 patterns (numpy) to a CUDA bfloat16 tensor (copy)."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    if out is None:
        return t.cuda()
    out.copy_(t)
    return out


def to_host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def rel_errors(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """|x_gpu - x_ref| / max(|x_ref|, 1e-3 * RMS(x_ref)): relative error with
    a floor so values that cross zero do not blow it up."""
    gpu = gpu.astype(np.float64)
    ref = ref.astype(np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    floor = max(1e-3 * rms, np.finfo(np.float32).tiny)
    return np.abs(gpu - ref) / np.maximum(np.abs(ref), floor)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (sign-magnitude order)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def compare_state(tag: str, gpu: dict, ref: dict, tol: float) -> dict:
    """Check fp32 w/m/v within ``tol`` (relative, with floor) and bf16 params
    within one ulp. Returns statistics (max error, bit-exact fraction)."""
    stats = {"case": tag, "tol": tol}
    for k in ("w", "m", "v"):
        e = rel_errors(gpu[k], ref[k])
        stats[f"{k}_max_rel"] = float(e.max()) if e.size else 0.0
        stats[f"{k}_bitexact"] = float(np.mean(gpu[k].view(np.uint32) == ref[k].view(np.uint32))) if e.size else 1.0
        assert stats[f"{k}_max_rel"] <= tol, (tag, k, stats)
    d = bf16_ulp_diff(gpu["p"], ref["p"])
    stats["p_max_ulp"] = int(d.max()) if d.size else 0
    stats["p_bitexact"] = float(np.mean(d == 0)) if d.size else 1.0
    assert stats["p_max_ulp"] <= 1, (tag, stats)
    log(stats)
    return stats


def log(record: dict) -> None:
    """Append a record to the file named by ZG_PARITY_LOG, if set."""
    path = os.environ.get("ZG_PARITY_LOG")
    if path:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")
