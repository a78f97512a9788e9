"""The norm pass taken bucket by bucket (Zero From Scratch, item 13).

Each bucket's sum of squares is added in submission order to a running fp64
sum; the last bucket makes the step's decision. The result must match the
whole-vector norm (same squares, different fp64 association: relative 1e-12),
and the step that follows must match the oracle. Bad bucket sequences are
refused before anything runs.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import to_dev_bf16, to_host_f32
from test_gpu_step import GpuRun, check_step
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu
L = 1024.0
F, LAST = zb.ZG_BUCKET_FIRST, zb.ZG_BUCKET_LAST


def split(n: int, size: int):
    """Contiguous buckets of `size` elements (multiples of 8), ragged tail last."""
    return [(lo, min(lo + size, n)) for lo in range(0, n, size)]


def bucket_norm(ctx, dev, buckets):
    for i, (lo, hi) in enumerate(buckets):
        flags = (F if i == 0 else 0) | (LAST if i == len(buckets) - 1 else 0)
        zb.zg_grad_norm_bucket(ctx, dev, lo, hi, L, flags)


@pytest.mark.parametrize("n,p,size", [(1_000_003, 8, 250_000), (65_549, 3, 65_549), (4099, 16, 1024),
                                      (300_000, 4, 8)])
def test_bucketed_norm_and_step(n, p, size):
    rng = np.random.default_rng(n + p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    run, whole = GpuRun(w0, p), GpuRun(w0, p)
    ref = oracle.OracleOptimizer(w0)
    buckets = split(n, size)
    for k in range(3):
        host = [synth.random_bf16(n, seed=700 + 10 * k + r, scale=(1e-3 if k != 1 else 0.5) * L) for r in range(p)]
        dev = [to_dev_bf16(h) for h in host]
        bucket_norm(run.ctx, dev, buckets)
        zb.zg_grad_norm(whole.ctx, dev, L)
        a, b = zb.zg_get_info(run.ctx), zb.zg_get_info(whole.ctx)
        assert a.found_inf == b.found_inf and abs(a.sumsq - b.sumsq) <= 1e-12 * b.sumsq
        zb.zg_shard_step(run.ctx, dev, L)
        zb.zg_shard_step(whole.ctx, dev, L)
        dec = ref.step(host, L)
        check_step(f"buckets n={n} p={p} size={size}", run, ref, dec, zb.zg_get_info(run.ctx), k + 1)


def test_bucketed_staged_gradient_equals_whole():
    n, p = 200_016, 8
    w0 = (np.random.default_rng(3).standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p)
    stage = torch.zeros(n, dtype=torch.float32, device="cuda")
    zb.zg_bind_grad_stage(run.ctx, stage)
    zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_STAGED)
    host = [synth.random_bf16(n, seed=90 + r, scale=1e-3 * L) for r in range(p)]
    bucket_norm(run.ctx, [to_dev_bf16(h) for h in host], split(n, 50_000))
    torch.cuda.synchronize()
    g = oracle.reduce_unscale(host, 0, n, oracle.inv_scale(L, p, 1))
    assert to_host_f32(stage).tobytes() == g.tobytes()


def test_bad_bucket_sequences_are_refused():
    n, p = 1024, 2
    run = GpuRun(np.zeros(n, np.float32), p)
    dev = [to_dev_bf16(synth.random_bf16(n, seed=r, scale=L)) for r in range(p)]
    bad = [
        [(8, 512, F)],                      # first bucket not at 0
        [(0, 512, 0)],                      # no sequence open
        [(0, 512, F), (520, 1024, LAST)],   # gap
        [(0, 512, F), (256, 1024, LAST)],   # overlap
        [(0, 512, F | LAST)],               # last bucket short of N
        [(0, 1024, F)],                     # ends at N without LAST
        [(0, 500, F), (500, 1024, LAST)],   # start not a multiple of 8
        [(0, 0, F)],                        # empty
        [(0, 2048, F | LAST)],              # past N
    ]
    for seq in bad:
        with pytest.raises(zb.ZgError) as e:
            for lo, hi, flags in seq:
                zb.zg_grad_norm_bucket(run.ctx, dev, lo, hi, L, flags)
        assert e.value.code == zb.ZG_ERR_INVALID_ARG, seq
    # a good sequence still works afterwards, and the step commits
    zb.zg_grad_norm_bucket(run.ctx, dev, 0, 512, L, F)
    zb.zg_grad_norm_bucket(run.ctx, dev, 512, 1024, L, LAST)
    zb.zg_shard_step(run.ctx, dev, L)
    info = zb.zg_get_info(run.ctx)
    assert info.status == 0 and info.step_t == 1
    # one bucket can be both first and last
    zb.zg_grad_norm_bucket(run.ctx, dev, 0, n, L, F | LAST)
    zb.zg_shard_step(run.ctx, dev, L)
    assert zb.zg_get_info(run.ctx).step_t == 2
