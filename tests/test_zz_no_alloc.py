"""zg_grad_norm_noalloc: the norm pass for callers that cannot allocate.

Some callers cannot call cudaMalloc (a framework allocator that already holds
nearly all device memory, a loop that cannot afford the synchronisation an
allocation may imply, a plug-in with no way to release memory it allocates).
For them the library offers a norm pass whose scratch is a fixed array
inside the library. These tests call it through the C ABI several times in a
row, on different sizes and rank counts, so every call runs on whatever the
previous one left in the shared array, and check each result:

- bit for bit against zg_grad_norm, the entry point that keeps its work
  array in a cudaMalloc'd workspace (same kernel, same exact summation);
- against the oracle's sum of squares of the reduced, unscaled gradient,
  within the norm tolerance of the other tests (relative 1e-5);
- on the degenerate sizes N = 1 and 7 and a ragged N = 65,549;
- with a planted +inf and a planted NaN, where the sum of squares must come
  out non-finite, followed by a finite call that must be right again.

Out-of-range sizes are refused with a message. The file is named to be
collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import to_dev_bf16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

L = 1024.0
NORM_TOL = 1e-5

# (N, P, seed, grad_average), run in this order
CASES = ((3_000_017, 8, 11, 1), (65_549, 3, 29, 1), (7, 2, 5, 1), (1, 1, 3, 1), (1_000_003, 16, 41, 1),
         (250_000, 5, 17, 0))


def _host(n: int, p: int, seed: int):
    return [synth.random_bf16(n, seed=seed + r, scale=1e-3 * L) for r in range(p)]


def _reference(grads, n: int, p: int, avg: int):
    ctx = zb.zg_init(n, p, zb.Hparams(grad_average=avg))
    zb.zg_grad_norm(ctx, grads, L)
    info = zb.zg_get_info(ctx)
    return info.sumsq, info.norm


def _noalloc(grads, n: int, p: int, avg: int = 1):
    lib = zb.lib()
    out = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    ptrs = (ctypes.c_void_p * p)(*[g.data_ptr() for g in grads])
    stream = torch.cuda.current_stream()
    rc = lib.zg_grad_norm_noalloc(ptrs, p, n, L, avg, out.data_ptr(), stream.cuda_stream)
    assert rc == zb.ZG_OK, lib.zg_last_error()
    stream.synchronize()
    return float(out[0]), float(out[1])


def _oracle_sumsq(host, n: int, p: int, avg: int) -> float:
    return oracle.sumsq(oracle.reduce_unscale(host, 0, n, oracle.inv_scale(L, p, avg)))


def test_noalloc_norm_equals_allocating_entry_point_and_oracle():
    for n, p, seed, avg in CASES:
        host = _host(n, p, seed)
        grads = [to_dev_bf16(h) for h in host]
        got_sumsq, got_norm = _noalloc(grads, n, p, avg)
        ref_sumsq, ref_norm = _reference(grads, n, p, avg)
        assert (got_sumsq, got_norm) == (ref_sumsq, ref_norm), (n, p, got_sumsq, ref_sumsq)
        want = _oracle_sumsq(host, n, p, avg)
        assert math.isfinite(got_sumsq) and abs(got_sumsq - want) <= NORM_TOL * want, (n, p, got_sumsq, want)
        assert got_norm == math.sqrt(got_sumsq)


def test_noalloc_norm_reports_inf_and_nan_then_recovers():
    n, p = 65_549, 4
    host = _host(n, p, 101)
    clean = [to_dev_bf16(h) for h in host]
    for pos, rank, bits in ((0, 2, 0x7F80), (n - 1, 0, 0x7FC0), (n // 2, p - 1, 0xFF80)):
        bad_host = [h.copy() for h in host]
        bad_host[rank][pos] = bits
        bad = [to_dev_bf16(h) for h in bad_host]
        got_sumsq, _ = _noalloc(bad, n, p)
        assert not math.isfinite(got_sumsq), (pos, rank, hex(bits), got_sumsq)
        assert not math.isfinite(_reference(bad, n, p, 1)[0])
        # the next finite call is not disturbed by what the bad one left behind
        got = _noalloc(clean, n, p)
        assert got == _reference(clean, n, p, 1)
        want = _oracle_sumsq(host, n, p, 1)
        assert abs(got[0] - want) <= NORM_TOL * want


def test_noalloc_refuses_out_of_range_sizes():
    lib = zb.lib()
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    one = (ctypes.c_void_p * 1)(g.data_ptr())
    for n, p, text in ((1 << 62, 1, b"N must be in"), (0, 1, b"N must be in"), (64, 17, b"P must be in"),
                       (64, 0, b"P must be in")):
        rc = lib.zg_grad_norm_noalloc(one, p, n, L, 1, out.data_ptr(), None)
        assert rc == zb.ZG_ERR_INVALID_ARG and text in lib.zg_last_error()
    assert np.all(out.cpu().numpy() == 0)  # nothing was launched
