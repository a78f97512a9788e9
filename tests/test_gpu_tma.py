"""The TMA-staged variant of the fused step: same results as the plain
variant bit for bit, parity with the oracle, and its bounded waits.

A wait limit of 0 makes the first wait of every CTA run out. The kernel must
then drain its own copies, write nothing, leave the step uncommitted, report
ZG_ERR_DEVICE_TIMEOUT through zg_get_info, and leave the context usable.
Small nonzero limits can run out after part of the state was written, which
must be reported as ZG_ERR_STATE_PARTIAL.
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


@pytest.mark.parametrize("n", [1, 7, 8, 2047, 2048, 2056, 65_549, 300_001])
@pytest.mark.parametrize("p", [1, 3, 8, 16])
def test_tma_edge_shapes(n, p):
    rng = np.random.default_rng(n + 7 * p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    tma, ldg = GpuRun(w0, p), GpuRun(w0, p)
    zb.zg_set_variant(tma.ctx, zb.ZG_VARIANT_TMA)
    ref = oracle.OracleOptimizer(w0)
    for k, host in enumerate(edge_sequence(n, p, seed=n * 13 + p), start=1):
        dev = [Guarded(n, torch.bfloat16) for _ in range(p)]
        for r in range(p):
            to_dev_bf16(host[r], dev[r].view)
        for run in (tma, ldg):
            zb.zg_step(run.ctx, [d.view for d in dev], L)
        info = zb.zg_get_info(tma.ctx)
        dec = ref.step(host, L)
        check_step(f"tma n={n} p={p}", tma, ref, dec, info, k)
        a, b = tma.state(), ldg.state()
        for key in a:
            assert a[key].tobytes() == b[key].tobytes(), (n, p, k, key)
    assert tma.guards_intact()


def test_tma_workload_matches_plain():
    w = synth.workload("flat16m_p8")
    total = synth.padded_len(w)
    w0 = torch.from_numpy(synth.init_weights(w))
    a = zb.ShardedAdamW(w.n, w.p, zb.Hparams(), w0)
    b = zb.ShardedAdamW(w.n, w.p, zb.Hparams(), w0)
    zb.zg_set_variant(a.ctx, zb.ZG_VARIANT_TMA)
    dev = [torch.empty(total, dtype=torch.bfloat16, device="cuda") for _ in range(w.p)]
    for k in range(1, 5):
        host = synth.step_grads(w, k)
        for r in range(w.p):
            to_dev_bf16(host[r], dev[r])
        a.step(dev, w.loss_scale)
        b.step(dev, w.loss_scale)
    for x, y in ((a.w, b.w), (a.m, b.m), (a.v, b.v), (a.params, b.params)):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                           y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
    assert a.info().step_t == b.info().step_t == 4


def test_wait_that_runs_out_reports_and_writes_nothing():
    n, p = 100_000, 4
    rng = np.random.default_rng(1)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p)
    zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_TMA)
    host = [synth.random_bf16(n, seed=90 + r, scale=1e-3 * L) for r in range(p)]
    dev = [to_dev_bf16(h) for h in host]
    zb.zg_step(run.ctx, dev, L)
    assert zb.zg_get_info(run.ctx).status == 0
    before = run.state()
    zb.zg_set_wait_limit(run.ctx, 0)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == zb.ZG_ERR_DEVICE_TIMEOUT and info.step_t == 1
    after = run.state()
    # the tail (fewer than 8 elements past the last tile) is not reached either
    for key in before:
        assert before[key].tobytes() == after[key].tobytes(), key
    assert zb.zg_get_info(run.ctx).status == 0  # cleared by the read
    # the context is still usable
    zb.zg_set_wait_limit(run.ctx, 4_000_000)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == 0 and info.step_t == 2
    ref = oracle.OracleOptimizer(w0)
    ref.step(host, L)
    ref.step(host, L)
    st = run.state()
    assert st["w"].tobytes() == ref.w.tobytes() or info.clip_coef != 1.0


@pytest.mark.parametrize("limit", [1, 8, 64, 512, 4096])
def test_wait_that_runs_out_mid_step_is_reported(limit):
    """A small nonzero wait limit can run out after some tiles are already
    written. Whatever happens, the status must say which state the buffers
    are in: a completed step equals the plain kernel's; ZG_ERR_DEVICE_TIMEOUT
    means nothing was written; ZG_ERR_STATE_PARTIAL means every element holds
    either its old or its new value. The step count stays in both failure
    cases, and after the state is restored the context steps normally."""
    n, p = (1 << 21) + 5, 8
    rng = np.random.default_rng(limit)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    host = [synth.random_bf16(n, seed=700 + r, scale=1e-3 * L) for r in range(p)]
    dev = [to_dev_bf16(h) for h in host]
    plain = GpuRun(w0, p)
    zb.zg_step(plain.ctx, dev, L)
    assert zb.zg_get_info(plain.ctx).status == 0
    new = plain.state()

    run = GpuRun(w0, p)
    zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_TMA)
    before = run.state()
    zb.zg_set_wait_limit(run.ctx, limit)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    after = run.state()
    assert info.status in (zb.ZG_OK, zb.ZG_ERR_DEVICE_TIMEOUT, zb.ZG_ERR_STATE_PARTIAL), info
    if info.status == zb.ZG_OK:
        assert info.step_t == 1
        for key in new:
            assert after[key].tobytes() == new[key].tobytes(), key
    elif info.status == zb.ZG_ERR_DEVICE_TIMEOUT:
        assert info.step_t == 0
        for key in before:
            assert after[key].tobytes() == before[key].tobytes(), key
    else:
        assert info.step_t == 0
        changed = 0
        for key in before:
            a, b, c = (x.view(np.uint32 if x.dtype == np.float32 else np.uint16) for x in (after[key], before[key],
                                                                                          new[key]))
            assert np.all((a == b) | (a == c)), key
            changed += int(np.count_nonzero(a != b))
        assert changed > 0
    assert run.guards_intact()
    log({"case": f"tma-mid-step-timeout/limit{limit}", "status": info.status})

    # restore the state, resume at step 0, and step with the default limit
    for key, arr in before.items():
        t = torch.from_numpy(arr.view(np.int16) if key == "p" else arr)
        run.bufs[key].view.copy_(t.view(torch.bfloat16) if key == "p" else t)
    zb.zg_set_step(run.ctx, 0)
    zb.zg_set_wait_limit(run.ctx, 4_000_000)
    zb.zg_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == 0 and info.step_t == 1
    again = run.state()
    for key in new:
        assert again[key].tobytes() == new[key].tobytes(), key
