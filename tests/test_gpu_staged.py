"""The staged variant: the norm pass stores the reduced fp32 gradient and the
step reads it. Results must equal the fused step bit for bit (both apply the
same fp32 operations to the same values), and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, to_dev_bf16, to_host_f32
from test_gpu_step import GpuRun, check_step, edge_sequence
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu
L = 1024.0


def _staged(run: GpuRun) -> Guarded:
    stage = Guarded(run.n, torch.float32)
    zb.zg_bind_grad_stage(run.ctx, stage.view)
    zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_STAGED)
    return stage


@pytest.mark.parametrize("n", [1, 7, 33, 2048, 65_549])
@pytest.mark.parametrize("p", [1, 4, 8, 16])
def test_staged_matches_fused_and_oracle(n, p):
    rng = np.random.default_rng(n + 3 * p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    staged, fused = GpuRun(w0, p), GpuRun(w0, p)
    stage = _staged(staged)
    ref = oracle.OracleOptimizer(w0)
    for k, host in enumerate(edge_sequence(n, p, seed=n * 7 + p), start=1):
        dev = [to_dev_bf16(h) for h in host]
        for run in (staged, fused):
            zb.zg_step(run.ctx, dev, L)
        info = zb.zg_get_info(staged.ctx)
        dec = ref.step(host, L)
        check_step(f"staged n={n} p={p}", staged, ref, dec, info, k)
        a, b = staged.state(), fused.state()
        for key in a:
            assert a[key].tobytes() == b[key].tobytes(), (n, p, k, key)
        if not dec.found_inf:  # the stage holds exactly the unscaled, averaged gradient
            g = oracle.reduce_unscale(host, 0, n, oracle.inv_scale(L, p, 1))
            assert to_host_f32(stage.view).tobytes() == g.tobytes()
    assert stage.intact() and staged.guards_intact()


def test_staged_needs_a_stage_buffer():
    ctx = zb.zg_init(64, 2)
    with pytest.raises(zb.ZgError) as e:
        zb.zg_set_variant(ctx, zb.ZG_VARIANT_STAGED)
    assert e.value.code == zb.ZG_ERR_NOT_BOUND


@pytest.mark.parametrize("n,p", [(33, 2), (65_549, 8), (4096, 16)])
def test_staged_mx_matches_fused_mx(n, p):
    """The MX path with the staged variant: the MX norm pass stores the
    reduced gradient (decoded products summed in rank order), the staged step
    reads it; identical bits to the fused MX step, and the oracle's step."""
    rng = np.random.default_rng(n * 5 + p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    staged, fused = GpuRun(w0, p), GpuRun(w0, p)
    stage = _staged(staged)
    ref = oracle.OracleOptimizer(w0)
    for k in range(4):
        host = [synth.random_bf16(n, seed=700 + 10 * k + r, scale=1e-3 if k != 1 else 1.0, dist="student_t")
                for r in range(p)]
        if k == 2:
            host[0][n // 3] = 0xFF80  # -inf: a skipped step
        enc = [oracle.mx_encode(h) for h in host]
        codes = [torch.from_numpy(c).cuda() for c, _ in enc]
        scales = [torch.from_numpy(s).cuda() for _, s in enc]
        for run in (staged, fused):
            zb.zg_step_mxfp8(run.ctx, codes, scales, 1.0)
        info = zb.zg_get_info(staged.ctx)
        dec = ref.step_mx([c for c, _ in enc], [s for _, s in enc], 1.0)
        check_step(f"staged mx n={n} p={p}", staged, ref, dec, info, k + 1)
        a, b = staged.state(), fused.state()
        for key in a:
            assert a[key].tobytes() == b[key].tobytes(), (n, p, k, key)
        if not dec.found_inf:
            g = oracle.mx_reduce_unscale([c for c, _ in enc], [s for _, s in enc], 0, n, oracle.inv_scale(1.0, p, 1))
            assert to_host_f32(stage.view).tobytes() == g.tobytes()
    assert stage.intact() and staged.guards_intact() and ref.t == 3
