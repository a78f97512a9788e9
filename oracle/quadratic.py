"""A tiny model whose every number can be worked by hand, for the gradient check.

TEST INFRASTRUCTURE ONLY (part of the oracle; see ``oracle/__init__.py``).

Zero From Scratch, item 17: a flat parameter vector and a gradient check
against finite differences. Item 6: data parallelism splits the batch, each
rank computes its gradient on its part, and the average of the rank gradients
equals the single-device gradient on the whole batch.

Model: f(w) = (1 / 2B) * sum_b || A_b w - y_b ||^2 over a batch of B samples,
with w a flat vector of n parameters, A_b a k x n matrix and y_b a k-vector.
Its gradient is (1 / B) * sum_b A_b^T (A_b w - y_b). Everything is float64.
"""
from __future__ import annotations

import numpy as np


def make_problem(n: int, k: int, batch: int, seed: int):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((batch, k, n))
    y = rng.standard_normal((batch, k))
    w = rng.standard_normal(n) * 0.1
    return a, y, w


def loss(w: np.ndarray, a: np.ndarray, y: np.ndarray) -> float:
    r = np.einsum("bkn,n->bk", a, w) - y
    return float(0.5 * np.sum(r * r) / a.shape[0])


def grad(w: np.ndarray, a: np.ndarray, y: np.ndarray) -> np.ndarray:
    r = np.einsum("bkn,n->bk", a, w) - y
    return np.einsum("bkn,bk->n", a, r) / a.shape[0]


def grad_fd(w: np.ndarray, a: np.ndarray, y: np.ndarray, h: float = 1e-5) -> np.ndarray:
    """Central differences, one coordinate at a time."""
    g = np.empty_like(w)
    for i in range(w.size):
        e = np.zeros_like(w)
        e[i] = h
        g[i] = (loss(w + e, a, y) - loss(w - e, a, y)) / (2.0 * h)
    return g


def dp_grads(w: np.ndarray, a: np.ndarray, y: np.ndarray, p: int) -> list[np.ndarray]:
    """Each of P ranks takes a contiguous 1/P of the batch and returns its own
    mean gradient over that part."""
    b = a.shape[0]
    assert b % p == 0
    part = b // p
    return [grad(w, a[r * part:(r + 1) * part], y[r * part:(r + 1) * part]) for r in range(p)]
