"""zg_grad_norm_noalloc: the norm pass for callers that cannot allocate.

Some callers cannot call cudaMalloc (a framework allocator that already holds
nearly all device memory, a loop that cannot afford the synchronisation an
allocation may imply, a plug-in with no way to release memory it allocates).
For them the library offers a norm pass whose scratch is a fixed array
inside the library. This test calls it through the C ABI twice in a row, on
different sizes and rank counts so the second call runs on whatever the first
left in the shared array, and checks each result against zg_grad_norm (the
entry point that uses a cudaMalloc'd workspace) within the norm tolerance of
the other tests (relative 1e-5). It also checks that out-of-range sizes are
refused with a message. The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import to_dev_bf16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

L = 1024.0
NORM_TOL = 1e-5


def _grads(n: int, p: int, seed: int):
    return [to_dev_bf16(synth.random_bf16(n, seed=seed + r, scale=1e-3 * L)) for r in range(p)]


def _reference(grads, n: int, p: int):
    ctx = zb.zg_init(n, p)
    zb.zg_grad_norm(ctx, grads, L)
    info = zb.zg_get_info(ctx)
    return info.sumsq, info.norm


def _noalloc(grads, n: int, p: int):
    lib = zb.lib()
    out = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    ptrs = (ctypes.c_void_p * p)(*[g.data_ptr() for g in grads])
    stream = torch.cuda.current_stream()
    rc = lib.zg_grad_norm_noalloc(ptrs, p, n, L, 1, out.data_ptr(), stream.cuda_stream)
    assert rc == zb.ZG_OK, lib.zg_last_error()
    stream.synchronize()
    return float(out[0]), float(out[1])


def test_noalloc_norm_matches_allocating_entry_point_twice():
    for n, p, seed in ((3_000_017, 8, 11), (65_549, 3, 29)):
        grads = _grads(n, p, seed)
        ref_sumsq, ref_norm = _reference(grads, n, p)
        got_sumsq, got_norm = _noalloc(grads, n, p)
        assert np.isfinite(got_sumsq)
        assert abs(got_sumsq - ref_sumsq) <= NORM_TOL * ref_sumsq, (n, p, got_sumsq, ref_sumsq)
        assert abs(got_norm - ref_norm) <= NORM_TOL * ref_norm, (n, p, got_norm, ref_norm)


def test_noalloc_refuses_out_of_range_sizes():
    lib = zb.lib()
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    one = (ctypes.c_void_p * 1)(g.data_ptr())
    for n, p, text in ((1 << 62, 1, b"N must be in"), (0, 1, b"N must be in"), (64, 17, b"P must be in"),
                       (64, 0, b"P must be in")):
        rc = lib.zg_grad_norm_noalloc(one, p, n, L, 1, out.data_ptr(), None)
        assert rc == zb.ZG_ERR_INVALID_ARG and text in lib.zg_last_error()
