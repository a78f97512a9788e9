"""The C ABI refuses memory of the wrong kind before it launches anything.

Every pointer is checked with cudaPointerGetAttributes: ordinary host memory
(here numpy arrays), pinned host memory where device memory is required, are
refused with ZG_ERR_INVALID_ARG and a message naming the argument, and no
kernel runs (the state and the step count are untouched). Pinned host memory
is accepted for w, m and v (optimizer state kept off the card). The calls go
straight to the C functions through ctypes, past the Python binding's own
checks, as a C caller would make them.
"""
import ctypes

import numpy as np
import pytest
import torch

from zero_sharded_mixed_flat_gb300 import binding as zb

pytestmark = pytest.mark.gpu

N, P, L = 4096, 2, 1024.0


def host_ptr(keep: list, nbytes: int) -> int:
    """A 16-byte aligned pointer into ordinary (pageable, unregistered) host
    memory; the array is kept alive in ``keep``."""
    a = np.zeros(nbytes + 64, dtype=np.uint8)
    keep.append(a)
    base = a.ctypes.data
    return base + (-base) % 16


def ptrs(*xs) -> ctypes.Array:
    return (ctypes.c_void_p * len(xs))(*xs)


def refused(rc: int, name: str) -> None:
    msg = zb.lib().zg_last_error().decode()
    assert rc == zb.ZG_ERR_INVALID_ARG, (rc, msg)
    assert name in msg, msg


@pytest.fixture
def bound():
    """A context with device state bound, device gradients, and its state."""
    ctx = zb.zg_init(N, P)
    s = zb.zg_shard_len(ctx)
    w = torch.randn(P * s, device="cuda") * 0.02
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    params = w.to(torch.bfloat16)
    zb.zg_bind(ctx, w, m, v, params)
    grads = [torch.randn(P * s, device="cuda").to(torch.bfloat16) for _ in range(P)]
    return ctx, (w, m, v, params), grads


def test_bind_checks_every_state_pointer(bound):
    ctx, (w, m, v, params), _ = bound
    lib, keep = zb.lib(), []
    h = host_ptr(keep, N * 4)
    refused(lib.zg_bind(ctx.handle, h, m.data_ptr(), v.data_ptr(), params.data_ptr()), "w ")
    refused(lib.zg_bind(ctx.handle, w.data_ptr(), m.data_ptr(), h, params.data_ptr()), "v ")
    pinned16 = torch.zeros(N, dtype=torch.bfloat16, pin_memory=True)
    refused(lib.zg_bind(ctx.handle, w.data_ptr(), m.data_ptr(), v.data_ptr(), pinned16.data_ptr()),
            "params is pinned host memory")
    # w, m and v may live in pinned host memory (optimizer state off the card)
    pw, pm, pv = (torch.zeros(N, dtype=torch.float32, pin_memory=True) for _ in range(3))
    assert lib.zg_bind(ctx.handle, pw.data_ptr(), pm.data_ptr(), pv.data_ptr(), params.data_ptr()) == zb.ZG_OK
    assert lib.zg_bind(ctx.handle, w.data_ptr(), m.data_ptr(), v.data_ptr(), params.data_ptr()) == zb.ZG_OK
    c = torch.zeros(N, dtype=torch.uint8, device="cuda")
    refused(lib.zg_bind_params_mxfp8(ctx.handle, h, c.data_ptr()), "codes")
    refused(lib.zg_bind_params_mxfp8(ctx.handle, c.data_ptr(), h), "scales")
    refused(lib.zg_bind_grad_stage(ctx.handle, h), "stage")


def test_steps_refuse_host_gradients_and_launch_nothing(bound):
    ctx, (w, m, v, params), grads = bound
    lib, keep = zb.lib(), []
    before = [t.clone() for t in (w, m, v, params)]
    h = host_ptr(keep, N * 2)
    pinned = torch.zeros(grads[0].numel(), dtype=torch.bfloat16, pin_memory=True)
    s = torch.cuda.current_stream().cuda_stream
    for bad, text in ((h, "grad_ptrs[1] is not memory CUDA knows"), (pinned.data_ptr(), "grad_ptrs[1] is pinned")):
        g = ptrs(grads[0].data_ptr(), bad)
        refused(lib.zg_step(ctx.handle, g, L, s), text)
        refused(lib.zg_grad_norm(ctx.handle, g, L, s), text)
        refused(lib.zg_shard_step(ctx.handle, g, L, s), text)
        refused(lib.zg_grad_norm_bucket(ctx.handle, g, 0, N, L, zb.ZG_BUCKET_FIRST | zb.ZG_BUCKET_LAST, s), text)
    info = zb.zg_get_info(ctx)
    assert info.status == 0 and info.step_t == 0
    for a, b in zip((w, m, v, params), before):
        assert torch.equal(a, b)
    # the device gradients still step (a refusal leaves nothing behind)
    zb.zg_step(ctx, grads, L)
    info = zb.zg_get_info(ctx)
    assert info.status == 0 and info.step_t == 1


def test_mx_gather_probe_and_noalloc_refuse_host_memory(bound):
    ctx, (w, m, v, params), grads = bound
    lib, keep = zb.lib(), []
    s = torch.cuda.current_stream().cuda_stream
    total = grads[0].numel()
    h = host_ptr(keep, total * 2)
    codes = [torch.zeros(total, dtype=torch.uint8, device="cuda") for _ in range(P)]
    scales = [torch.zeros(total // 32, dtype=torch.uint8, device="cuda") for _ in range(P)]
    refused(lib.zg_quant_mxfp8(h, N, codes[0].data_ptr(), scales[0].data_ptr(), s), "in ")
    refused(lib.zg_quant_mxfp8(grads[0].data_ptr(), N, h, scales[0].data_ptr(), s), "codes")
    refused(lib.zg_quant_mxfp8(grads[0].data_ptr(), N, codes[0].data_ptr(), h, s), "scales")
    refused(lib.zg_step_mxfp8(ctx.handle, ptrs(codes[0].data_ptr(), h), ptrs(*[x.data_ptr() for x in scales]), 1.0, s),
            "codes[1]")
    refused(lib.zg_step_mxfp8(ctx.handle, ptrs(*[x.data_ptr() for x in codes]), ptrs(scales[0].data_ptr(), h), 1.0, s),
            "scales[1]")
    out = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    sh = zb.zg_shard_len(ctx)
    shards = ptrs(params.data_ptr(), params.data_ptr() + sh * 2)
    refused(lib.zg_gather_params(ctx.handle, shards, 0, N, h, s), "out")
    refused(lib.zg_gather_params(ctx.handle, ptrs(params.data_ptr(), h), 0, N, out.data_ptr(), s), "shards[1]")
    refused(lib.zg_gather_params_dma(ctx.handle, shards, 0, N, h, s), "out")
    refused(lib.zg_gather_params_mxfp8(ctx.handle, ptrs(codes[0].data_ptr(), h), ptrs(*[x.data_ptr() for x in scales]),
                                       0, N, out.data_ptr(), s), "codes[1]")
    refused(lib.zg_probe_copy(h, out.data_ptr(), 1024, s), "src")
    refused(lib.zg_probe_copy(out.data_ptr(), h, 1024, s), "dst")
    res = torch.zeros(2, dtype=torch.float64, device="cuda")
    refused(lib.zg_grad_norm_noalloc(ptrs(grads[0].data_ptr(), h), P, N, L, 1, res.data_ptr(), s), "grad_ptrs[1]")
    refused(lib.zg_grad_norm_noalloc(ptrs(*[g.data_ptr() for g in grads]), P, N, L, 1, h, s), "out")
    info = zb.zg_get_info(ctx)
    assert info.status == 0 and info.step_t == 0
