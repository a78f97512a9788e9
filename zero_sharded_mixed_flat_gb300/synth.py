"""Seeded synthetic inputs for the optimizer step.

This module is the one thing the CUDA path's tests and the oracle share: it
draws initial master weights and per-rank bf16 gradients, and holds none of
the step's arithmetic. Every value is a pure function of
(seed, stream, step, rank, chunk), so any slice of any buffer can be drawn
again on its own, in any order and on any thread, with the same bits.

Streams: 0 = initial master weights, 1 = gradients of (step, rank),
2 = per-tensor gradient scales of a step, 3 = where the injected inf goes.

Workloads (sizes and distributions from the optimizer-step workloads this
library is measured on; the pages describe no dataset, so all inputs are
synthetic):
  flat65k_p4      N = 65,536, P = 4, grads N(0, 1e-3) x 1024, 10 steps
  flat16m_p8      N = 2^24, P = 8, as above, 20 steps, +inf at step 7 rank 3
  gpt2small_p8    N = 124,439,808 (the 148 GPT-2-small tensors in module
                  order), P = 8, one log-uniform[1e-5, 1e-2] scale per tensor
                  per step, loss scale 65,536, 5 steps; 25M-element buckets
  flat3b_p8       N = 3e9, P = 8, grads N(0, 1e-3) x 1024, 3 steps
  mxfp8_128m_p8   N = 2^27, P = 8, Student-t(3) x 1e-3, loss scale 1, MXFP8
Master weights start N(0, 0.02); m and v start at zero.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

CHUNK = 1 << 20  # elements per independently seeded chunk

STREAM_W, STREAM_GRAD, STREAM_SIGMA, STREAM_INF = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    p: int
    loss_scale: float
    steps: int
    dist: str  # "normal" | "per_tensor" | "student_t"
    seed: int
    sigma: float = 1e-3
    mx: bool = False
    inf_step: int | None = None  # 1-based step that carries an injected +inf
    inf_rank: int | None = None


WORKLOADS = {
    w.name: w
    for w in (
        Workload("flat65k_p4", 65_536, 4, 1024.0, 10, "normal", 0x5A0E0001),
        Workload("flat16m_p8", 1 << 24, 8, 1024.0, 20, "normal", 0x5A0E0002, inf_step=7, inf_rank=3),
        Workload("gpt2small_p8", 124_439_808, 8, 65536.0, 5, "per_tensor", 0x5A0E0003),
        Workload("flat3b_p8", 3_000_000_000, 8, 1024.0, 3, "normal", 0x5A0E0004),
        Workload("mxfp8_128m_p8", 1 << 27, 8, 1.0, 5, "student_t", 0x5A0E0005, mx=True),
    )
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    if overrides:
        w = Workload(**{**w.__dict__, **overrides})
    return w


# ------------------------------------------------------------ GPT-2 small

def gpt2_small_tensors() -> list[tuple[str, int]]:
    """The parameter tensors of GPT-2 small (d=768, 12 layers, vocabulary
    50,257, context 1,024, tied output embedding) in module order: 148
    tensors, 124,439,808 numbers."""
    d, layers, vocab, ctx = 768, 12, 50257, 1024
    out = [("wte", vocab * d), ("wpe", ctx * d)]
    for i in range(layers):
        out += [
            (f"h{i}.ln_1.weight", d), (f"h{i}.ln_1.bias", d),
            (f"h{i}.attn.c_attn.weight", d * 3 * d), (f"h{i}.attn.c_attn.bias", 3 * d),
            (f"h{i}.attn.c_proj.weight", d * d), (f"h{i}.attn.c_proj.bias", d),
            (f"h{i}.ln_2.weight", d), (f"h{i}.ln_2.bias", d),
            (f"h{i}.mlp.c_fc.weight", d * 4 * d), (f"h{i}.mlp.c_fc.bias", 4 * d),
            (f"h{i}.mlp.c_proj.weight", 4 * d * d), (f"h{i}.mlp.c_proj.bias", d),
        ]
    out += [("ln_f.weight", d), ("ln_f.bias", d)]
    return out


def buckets(n: int, size: int = 25_000_000) -> list[tuple[int, int]]:
    """Contiguous gradient buckets [lo, hi) of ``size`` elements, ragged tail last."""
    return [(lo, min(lo + size, n)) for lo in range(0, n, size)]


def tensor_sigmas(w: Workload, step: int) -> np.ndarray:
    """One gradient scale per tensor for this step, log-uniform on [1e-5, 1e-2],
    shared by all ranks."""
    rng = _rng(w.seed, STREAM_SIGMA, step, 0, 0)
    k = len(gpt2_small_tensors())
    return np.exp(rng.uniform(math.log(1e-5), math.log(1e-2), size=k))


# ------------------------------------------------------------ generators

def _rng(seed: int, stream: int, step: int, rank: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, step, rank, chunk])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunked(lo: int, hi: int, make_chunk, dtype, out: np.ndarray | None = None) -> np.ndarray:
    """Assemble [lo, hi) from whole seeded chunks, drawing chunks in parallel,
    into ``out`` (hi - lo elements of ``dtype``) or a new array."""
    if out is None:
        out = np.empty(max(hi - lo, 0), dtype=dtype)
    elif out.dtype != dtype or out.shape != (max(hi - lo, 0),):
        raise ValueError(f"out must be {max(hi - lo, 0)} elements of {np.dtype(dtype)}")
    if hi <= lo:
        return out
    first, last = lo // CHUNK, (hi - 1) // CHUNK

    def fill(c: int) -> None:
        data = make_chunk(c)
        a, b = max(lo, c * CHUNK), min(hi, (c + 1) * CHUNK)
        out[a - lo:b - lo] = data[a - c * CHUNK:b - c * CHUNK]

    chunks = range(first, last + 1)
    if len(chunks) == 1:
        fill(first)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, chunks))
    return out


def init_weights(w: Workload, lo: int = 0, hi: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Initial fp32 master weights for flat indices [lo, hi), N(0, 0.02)
    (into ``out``, float32, hi - lo elements, when given)."""
    hi = w.n if hi is None else hi

    def chunk(c: int) -> np.ndarray:
        return _rng(w.seed, STREAM_W, 0, 0, c).standard_normal(CHUNK, dtype=np.float32) * np.float32(0.02)

    return _chunked(lo, hi, chunk, np.float32, out)


def _grad_chunk_maker(w: Workload, step: int, rank: int):
    """chunk index -> that chunk's unscaled float32 gradient values."""
    if w.dist == "per_tensor":
        sizes = np.array([s for _, s in gpt2_small_tensors()], dtype=np.int64)
        starts = np.concatenate([[0], np.cumsum(sizes)])
        sig = tensor_sigmas(w, step)

    def chunk(c: int) -> np.ndarray:
        rng = _rng(w.seed, STREAM_GRAD, step, rank, c)
        if w.dist == "normal":
            return rng.standard_normal(CHUNK, dtype=np.float32) * np.float32(w.sigma)
        if w.dist == "student_t":
            z = rng.standard_normal(CHUNK)
            chi = rng.chisquare(3.0, CHUNK)
            return (z / np.sqrt(chi / 3.0) * w.sigma).astype(np.float32)
        if w.dist == "per_tensor":
            z = rng.standard_normal(CHUNK, dtype=np.float32)
            idx = np.arange(c * CHUNK, (c + 1) * CHUNK, dtype=np.int64)
            seg = np.clip(np.searchsorted(starts, idx, side="right") - 1, 0, len(sig) - 1)
            return z * sig[seg].astype(np.float32)
        raise ValueError(w.dist)

    return chunk


def grad_values(w: Workload, step: int, rank: int, lo: int = 0, hi: int | None = None) -> np.ndarray:
    """Rank ``rank``'s unscaled gradient values for step ``step`` (1-based) on
    [lo, hi), as float32, before the loss scale and bf16 storage."""
    hi = w.n if hi is None else hi
    return _chunked(lo, hi, _grad_chunk_maker(w, step, rank), np.float32)


def inf_index(w: Workload, step: int) -> int | None:
    """Flat index that carries +inf at the injection step, else None."""
    if w.inf_step is None or step != w.inf_step:
        return None
    return int(_rng(w.seed, STREAM_INF, step, 0, 0).integers(0, w.n))


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns by the library cast (round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def grads_bf16(w: Workload, step: int, rank: int, lo: int = 0, hi: int | None = None,
               loss_scale: float | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """The stored gradient: bf16(f32(x) * L) on [lo, hi) (indices at or past
    N are padding and read as +0), plus the injected +inf, if any. Each
    chunk is drawn, scaled and cast on its own worker thread. ``out`` (uint16,
    hi - lo elements), when given, receives the values instead of a new array."""
    hi = w.n if hi is None else hi
    ls = np.float32(w.loss_scale if loss_scale is None else loss_scale)
    make = _grad_chunk_maker(w, step, rank)

    def chunk(c: int) -> np.ndarray:
        x = make(c)
        x *= ls
        if (c + 1) * CHUNK > w.n:
            x[max(0, w.n - c * CHUNK):] = 0.0
        return _to_bf16_bits(x)

    out = _chunked(lo, hi, chunk, np.uint16, out)
    k = inf_index(w, step)
    if k is not None and rank == w.inf_rank and lo <= k < hi:
        out[k - lo] = 0x7F80
    return out


def padded_len(w: Workload) -> int:
    """P * S: the buffer length, with S = ceil(N/P) rounded up to 32."""
    s = -(-w.n // w.p)
    s = -(-s // 32) * 32
    return w.p * s


def step_grads(w: Workload, step: int, loss_scale: float | None = None) -> list[np.ndarray]:
    """All P gradient buffers of a step, each P * S long (padding zero)."""
    total = padded_len(w)
    return [grads_bf16(w, step, r, 0, total, loss_scale) for r in range(w.p)]


def random_bf16(n: int, seed: int, scale: float = 1.0, dist: str = "normal") -> np.ndarray:
    """A free-standing seeded bf16 vector (for small edge-case tests)."""
    rng = _rng(seed, 9, 0, 0, 0)
    if dist == "normal":
        x = rng.standard_normal(n).astype(np.float32) * np.float32(scale)
    elif dist == "student_t":
        x = (rng.standard_normal(n) / np.sqrt(rng.chisquare(3.0, n) / 3.0) * scale).astype(np.float32)
    elif dist == "logspread":
        # magnitudes spread over many binades, random signs
        x = (np.exp(rng.uniform(-60, 60, n)) * rng.choice([-1.0, 1.0], n) * scale).astype(np.float32)
    else:
        raise ValueError(dist)
    return _to_bf16_bits(x)
