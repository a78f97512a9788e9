"""Ring collectives on P in-memory ranks, with hop and byte counting.

TEST INFRASTRUCTURE ONLY (part of the oracle; see ``oracle/__init__.py``).

Zero From Scratch, item 7: all-reduce, reduce-scatter and all-gather, and the
identity all-reduce = all-gather(reduce-scatter(x)). Item 8 and item 17: the
collectives are charged at ring cost, where one all-reduce takes 2(P - 1)
hops (six at P = 4). Each function moves whole chunks between ranks one hop at
a time, so every message is counted.

Rank r owns chunk r of the flat vector (the same contiguous split as the
optimizer's shards). In the ring reduce-scatter, the partial of chunk c starts
at rank c+1 and travels forward; after P - 1 hops it reaches rank c with all P
contributions added, in the rotated order c+1, c+2, ..., c.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Wire:
    """What the ring moved: hops (communication rounds) and elements sent per rank."""

    hops: int = 0
    sent: list = field(default_factory=list)

    def send(self, rank: int, n: int) -> None:
        self.sent[rank] += n


def _chunks(m: int, p: int) -> list[tuple[int, int]]:
    s = -(-m // p)
    return [(min(r * s, m), min((r + 1) * s, m)) for r in range(p)]


def reduce_scatter(xs: list[np.ndarray], wire: Wire | None = None) -> list[np.ndarray]:
    """Ring reduce-scatter of P equal-length vectors: returns, for each rank r,
    the sum over ranks of chunk r. P - 1 hops; each rank sends (P-1)/P of M."""
    p = len(xs)
    m = xs[0].size
    wire = wire if wire is not None else Wire(sent=[0] * p)
    if not wire.sent:
        wire.sent = [0] * p
    bounds = _chunks(m, p)
    # partial[r][c]: rank r's running partial of chunk c
    partial = [[xs[r][lo:hi].copy() for (lo, hi) in bounds] for r in range(p)]
    for h in range(p - 1):
        msgs = []
        for r in range(p):
            c = (r - h - 1) % p
            msgs.append((r, (r + 1) % p, c, partial[r][c].copy()))
            wire.send(r, partial[r][c].size)
        for _src, dst, c, data in msgs:
            partial[dst][c] = data + partial[dst][c]
        wire.hops += 1
    return [partial[r][r] for r in range(p)]


def all_gather(shards: list[np.ndarray], wire: Wire | None = None) -> list[np.ndarray]:
    """Ring all-gather: every rank ends with the concatenation of all shards.
    P - 1 hops; each rank sends (P-1)/P of M."""
    p = len(shards)
    wire = wire if wire is not None else Wire(sent=[0] * p)
    if not wire.sent:
        wire.sent = [0] * p
    have = [{r: shards[r].copy()} for r in range(p)]
    for h in range(p - 1):
        msgs = []
        for r in range(p):
            c = (r - h) % p
            msgs.append(((r + 1) % p, c, have[r][c].copy()))
            wire.send(r, have[r][c].size)
        for dst, c, data in msgs:
            have[dst][c] = data
        wire.hops += 1
    return [np.concatenate([have[r][c] for c in range(p)]) for r in range(p)]


def all_reduce(xs: list[np.ndarray], wire: Wire | None = None) -> list[np.ndarray]:
    """Ring all-reduce, built as reduce-scatter followed by all-gather."""
    wire = wire if wire is not None else Wire(sent=[0] * len(xs))
    return all_gather(reduce_scatter(xs, wire), wire)


def all_reduce_direct(xs: list[np.ndarray]) -> list[np.ndarray]:
    """All-reduce by its definition: every rank receives the elementwise sum."""
    total = np.zeros_like(xs[0])
    for x in xs:
        total = total + x
    return [total.copy() for _ in xs]
