"""The one-launch variant of the bf16 step (ZG_VARIANT_SINGLE): the norm pass,
a grid-wide barrier and the fused step pass in one cooperative launch.

Its norm is the same exact sum the two-launch norm pass takes (warp chunks,
the fixed-point total), so the sum of squares, the decision and the state it
writes must be the two-launch variant's bit for bit, and match the oracle
within the stated tolerances (bit for bit when the clip factors agree) on the
edge sequence of ordinary, clipped, +inf and NaN steps.
The barrier's wait is bounded: a limit of 0 makes every block give up before
storing anything (ZG_ERR_DEVICE_TIMEOUT, state untouched, step count kept);
small limits may also give ZG_ERR_STATE_PARTIAL, with every element either
old or new. Either way the context keeps working.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, log, to_dev_bf16
from test_gpu_step import GpuRun, check_step, edge_sequence
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu
L = 1024.0


@pytest.mark.parametrize("n", [1, 7, 8, 2047, 65_549, 300_001])
@pytest.mark.parametrize("p", [1, 3, 8, 16])
def test_single_launch_edge_shapes(n, p):
    rng = np.random.default_rng(n + 11 * p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    one, two = GpuRun(w0, p), GpuRun(w0, p)
    zb.zg_set_variant(one.ctx, zb.ZG_VARIANT_SINGLE)
    ref = oracle.OracleOptimizer(w0)
    for k, host in enumerate(edge_sequence(n, p, seed=n * 17 + p), start=1):
        dev = [Guarded(n, torch.bfloat16) for _ in range(p)]
        for r in range(p):
            to_dev_bf16(host[r], dev[r].view)
        for run in (one, two):
            zb.zg_step(run.ctx, [d.view for d in dev], L)
        info, info2 = zb.zg_get_info(one.ctx), zb.zg_get_info(two.ctx)
        dec = ref.step(host, L)
        check_step(f"single n={n} p={p}", one, ref, dec, info, k)
        assert info.found_inf == info2.found_inf and info.step_t == info2.step_t
        if not dec.found_inf:
            assert (info.sumsq, info.clip_coef) == (info2.sumsq, info2.clip_coef), (n, p, k, info, info2)
        a, b = one.state(), two.state()
        for key in a:
            assert a[key].tobytes() == b[key].tobytes(), (n, p, k, key)
        assert all(d.intact() for d in dev)
    assert one.guards_intact()


def test_single_launch_workload_matches_two_launches():
    """flat16m_p8's first eight steps (step 7 carries the injected +inf and
    is skipped) through both variants: the same decisions and the same
    state bits."""
    w = synth.workload("flat16m_p8")
    total = synth.padded_len(w)
    w0 = torch.from_numpy(synth.init_weights(w))
    a = zb.ShardedAdamW(w.n, w.p, zb.Hparams(), w0)
    b = zb.ShardedAdamW(w.n, w.p, zb.Hparams(), w0)
    zb.zg_set_variant(a.ctx, zb.ZG_VARIANT_SINGLE)
    dev = [torch.empty(total, dtype=torch.bfloat16, device="cuda") for _ in range(w.p)]
    for k in range(1, 9):
        for r, h in enumerate(synth.step_grads(w, k)):
            to_dev_bf16(h, dev[r])
        a.step(dev, w.loss_scale)
        b.step(dev, w.loss_scale)
        ia, ib = a.info(), b.info()
        assert ia.status == ib.status == 0 and ia.found_inf == ib.found_inf == (k == 7)
        assert ia.clip_coef == ib.clip_coef and ia.step_t == ib.step_t
        if not ia.found_inf:
            assert ia.norm == ib.norm
    for x, y in ((a.w, b.w), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a.params.view(torch.int16), b.params.view(torch.int16))
    assert a.info().step_t == 7


def test_single_launch_barrier_limit_zero_writes_nothing():
    n, p = 1 << 20, 8
    rng = np.random.default_rng(2)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p)
    zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_SINGLE)
    host = [synth.random_bf16(n, seed=300 + r, scale=1e-3 * L) for r in range(p)]
    dev = [to_dev_bf16(h) for h in host]
    zb.zg_step(run.ctx, dev, L)
    assert zb.zg_get_info(run.ctx).status == 0
    before = run.state()
    zb.zg_set_wait_limit(run.ctx, 0)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == zb.ZG_ERR_DEVICE_TIMEOUT and info.step_t == 1
    after = run.state()
    for key in before:
        assert before[key].tobytes() == after[key].tobytes(), key
    assert zb.zg_get_info(run.ctx).status == 0  # cleared by the read
    # the norm was consumed: a shard step on its own is refused as stale
    zb.zg_shard_step(run.ctx, dev, L)
    assert zb.zg_get_info(run.ctx).status == zb.ZG_ERR_STALE_NORM
    # the context keeps working
    zb.zg_set_wait_limit(run.ctx, 4_000_000)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == 0 and info.step_t == 2
    ref = oracle.OracleOptimizer(w0)
    ref.step(host, L)
    dec = ref.step(host, L)
    st = run.state()
    assert st["w"].tobytes() == ref.w.tobytes() or info.clip_coef != dec.clip


@pytest.mark.parametrize("limit", [1, 2, 16])
def test_single_launch_small_limits_report_the_state(limit):
    n, p = (1 << 21) + 3, 8
    rng = np.random.default_rng(100 + limit)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    host = [synth.random_bf16(n, seed=900 + r, scale=1e-3 * L) for r in range(p)]
    dev = [to_dev_bf16(h) for h in host]
    plain = GpuRun(w0, p)
    zb.zg_step(plain.ctx, dev, L)
    new = plain.state()
    clip_plain = zb.zg_get_info(plain.ctx).clip_coef
    run = GpuRun(w0, p)
    zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_SINGLE)
    before = run.state()
    zb.zg_set_wait_limit(run.ctx, limit)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    after = run.state()
    assert info.status in (zb.ZG_OK, zb.ZG_ERR_DEVICE_TIMEOUT, zb.ZG_ERR_STATE_PARTIAL), info
    if info.status == zb.ZG_OK:
        assert info.step_t == 1
        if info.clip_coef == clip_plain:
            for key in new:
                assert after[key].tobytes() == new[key].tobytes(), key
    elif info.status == zb.ZG_ERR_DEVICE_TIMEOUT:
        assert info.step_t == 0
        for key in before:
            assert after[key].tobytes() == before[key].tobytes(), key
    else:
        assert info.step_t == 0
        for key in before:
            a, b, c = (x.view(np.uint32 if x.dtype == np.float32 else np.uint16) for x in (after[key], before[key],
                                                                                          new[key]))
            assert np.all((a == b) | (a == c)), key
    log({"case": f"single-launch-barrier/limit{limit}", "status": info.status})
    # restore, resume at 0, step with the default limit
    for key, arr in before.items():
        t = torch.from_numpy(arr.view(np.int16) if key == "p" else arr)
        run.bufs[key].view.copy_(t.view(torch.bfloat16) if key == "p" else t)
    zb.zg_set_step(run.ctx, 0)
    zb.zg_set_wait_limit(run.ctx, 4_000_000)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == 0 and info.step_t == 1
    assert run.guards_intact()


def test_single_launch_refuses_mx_parameters():
    ctx = zb.zg_init(4096, 2)
    s = zb.zg_shard_len(ctx)
    w = torch.zeros(2 * s, device="cuda")
    zb.zg_bind(ctx, w, torch.zeros_like(w), torch.zeros_like(w), w.to(torch.bfloat16))
    codes = torch.zeros(2 * s, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(2 * s // 32, dtype=torch.uint8, device="cuda")
    zb.zg_bind_params_mxfp8(ctx, codes, scales)
    with pytest.raises(zb.ZgError):
        zb.zg_set_variant(ctx, zb.ZG_VARIANT_SINGLE)
    zb.zg_bind_params_mxfp8(ctx, None, None)
    zb.zg_set_variant(ctx, zb.ZG_VARIANT_SINGLE)
    with pytest.raises(zb.ZgError):
        zb.zg_bind_params_mxfp8(ctx, codes, scales)
