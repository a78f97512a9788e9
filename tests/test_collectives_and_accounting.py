"""Pins on the pages' own figures and on the collective identity.

Zero From Scratch, items 1, 3, 8, 9, 14 and 18 print the figures in
``golden/page_figures.json``; item 7 states all-reduce = all-gather after
reduce-scatter; item 17 asks for a gradient check against finite differences;
item 6 says the averaged data-parallel gradient matches a single device.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import quadratic, ring
from zero_sharded_mixed_flat_gb300 import accounting as acc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
GIB = 2 ** 30


def test_sixteen_bytes_per_weight():
    assert acc.bytes_per_weight() == GOLD["bytes_per_weight"]["value"]
    assert acc.PARAM_BF16 == GOLD["bytes_per_weight"]["versus"]
    assert len(GOLD["state_parts"]["value"]) + 1 == 5  # the weight itself + four parts


def test_replicated_state_of_the_30b_model():
    n = GOLD["model_params"]["value"]
    stage0 = acc.per_gpu_bytes(n, 8, acc.STAGES[0]) / GIB
    assert round(stage0) == GOLD["replicated_state_gib"]["value"]
    # every stage but the third leaves more than one card's worth on each of 8 GPUs
    card = GOLD["card_memory_gb"]["value"] * 1e9
    fits = {s: acc.per_gpu_bytes(n, 8, acc.STAGES[s]) <= card for s in range(4)}
    assert fits == {0: False, 1: False, 2: False, 3: True}
    assert len(acc.STAGES) - 1 == GOLD["stages"]["value"]
    assert len(acc.Stage.__dataclass_fields__) == GOLD["flags"]["value"]


def test_replicated_floor():
    n = 30e9
    for s, stage in acc.STAGES.items():
        floor = acc.replicated_floor_bytes(n, stage)
        # the per-GPU bytes approach the floor as P grows and never go below it
        assert acc.per_gpu_bytes(n, 10 ** 6, stage) >= floor
        assert acc.per_gpu_bytes(n, 10 ** 6, stage) - floor < n * 16 / 10 ** 5
    assert acc.replicated_floor_bytes(n, acc.STAGES[3]) == 0


def test_mxfp8_savings():
    assert round(100 * acc.mxfp8_stored_state_saving()) == GOLD["mxfp8_state_saving_pct"]["value"]
    assert abs(acc.mxfp8_wire_saving() - GOLD["mxfp8_wire_saving"]["value"]) < 0.02


def test_fusion_trips():
    assert acc.unfused_memory_trips(GOLD["unfused_trips"]["ops"]) == GOLD["unfused_trips"]["value"]
    assert acc.fused_memory_trips(3) == 2


@pytest.mark.parametrize("p", range(1, 9))
def test_ring_all_reduce_identity(p):
    """AR = AG(RS(x)) by brute force on integer values (every order exact),
    with the hop count and bytes of a ring."""
    rng = np.random.default_rng(p)
    for m in (p, 8 * p, 64 if 64 % p == 0 else 8 * p):
        xs = [rng.integers(-1000, 1000, size=m).astype(np.float32) for _ in range(p)]
        wire = ring.Wire(sent=[0] * p)
        rs = ring.reduce_scatter(xs, wire)
        assert wire.hops == acc.ring_hops(p, "reduce_scatter")
        ag = ring.all_gather(rs, wire)
        assert wire.hops == acc.ring_hops(p, "all_reduce")
        direct = ring.all_reduce_direct(xs)
        for r in range(p):
            assert np.array_equal(ag[r], direct[r])
        for r in range(p):
            assert wire.sent[r] == acc.ring_bytes_sent_per_rank(m, p, "all_reduce")
    if p == 4:
        assert wire.hops == GOLD["ring_hops"]["value"]


@pytest.mark.parametrize("p", [1, 2, 3, 4, 8])
def test_ring_shard_equals_oracle_reduce(p):
    """Rank r's reduce-scatter output is the oracle's reduce over shard r
    (integer-valued bf16 gradients, so every order of addition is exact)."""
    rng = np.random.default_rng(10 + p)
    n = 333
    s = oracle.shard_len(n, p)
    ints = rng.integers(-100, 100, size=(p, p * s)).astype(np.float32)
    ints[:, n:] = 0
    grads = [(ints[r].view(np.uint32) >> 16).astype(np.uint16) for r in range(p)]
    rs = ring.reduce_scatter([ints[r] for r in range(p)])
    inv = oracle.inv_scale(1.0, p, 0)
    for r in range(p):
        lo, hi = min(r * s, n), min((r + 1) * s, n)
        g = oracle.reduce_unscale(grads, lo, hi, inv)
        assert np.array_equal(g, rs[r][: hi - lo])


def test_finite_difference_gradient_check():
    a, y, w = quadratic.make_problem(n=12, k=5, batch=8, seed=0)
    g = quadratic.grad(w, a, y)
    fd = quadratic.grad_fd(w, a, y, h=1e-5)
    assert np.max(np.abs(g - fd)) <= 1e-7 * np.max(np.abs(g))


@pytest.mark.parametrize("p", [1, 2, 4, 8])
def test_data_parallel_average_matches_single_device(p):
    a, y, w = quadratic.make_problem(n=10, k=3, batch=16, seed=1)
    full = quadratic.grad(w, a, y)
    avg = sum(quadratic.dp_grads(w, a, y, p)) / p
    assert np.allclose(avg, full, rtol=1e-13, atol=1e-15)


def test_kernel_byte_formulas():
    assert acc.shard_step_bytes_per_param(8) == 42 and acc.shard_step_bytes_per_param(4) == 34
    assert acc.grad_norm_bytes_per_param(8) == 16
    assert acc.mx_shard_step_bytes_per_param(8) == 8 * (1 + 1 / 32) + 26
    r = acc.resident_bytes(3_000_000_000, 8, 375_000_000)
    assert r == {"state": 36e9, "params": 6e9, "grads": 48e9}
