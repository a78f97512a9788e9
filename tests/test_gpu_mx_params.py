"""Parameters stored as MXFP8 (Zero From Scratch, item 14: MXFP8 on stored
state). With MX parameter buffers bound, each step encodes the updated fp32
master weights per 32-element block instead of writing bf16. w, m and v must
match the oracle as before, and the codes and scale bytes must equal the
oracle's encoding of the oracle's weights bit for bit; the bf16 buffer is left
alone, and a skipped step writes nothing."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, rel_errors, to_dev_bf16, to_host_f32, to_host_u16
from test_gpu_step import GpuRun, edge_sequence
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu
L = 1024.0


class MxRun(GpuRun):
    def __init__(self, w0, p, variant=None):
        super().__init__(w0, p)
        self.codes = Guarded(self.n, torch.uint8)
        self.scales = Guarded((self.n + 31) // 32, torch.uint8)
        if variant == "staged":
            self.stage = torch.zeros(self.n, dtype=torch.float32, device="cuda")
            zb.zg_bind_grad_stage(self.ctx, self.stage)
            zb.zg_set_variant(self.ctx, zb.ZG_VARIANT_STAGED)
        zb.zg_bind_params_mxfp8(self.ctx, self.codes.view, self.scales.view)
        self.p_before = to_host_u16(self.bufs["p"].view).copy()

    def check(self, tag, ref, dec, info):
        assert info.status == 0 and info.found_inf == dec.found_inf and info.step_t == ref.t, (tag, info)
        st = self.state()
        same = info.clip_coef == dec.clip
        for k in ("w", "m", "v"):
            if same:
                assert st[k].tobytes() == getattr(ref, k).tobytes(), (tag, k)
            else:
                assert rel_errors(st[k], getattr(ref, k)).max() <= 2e-6 * max(ref.t, 1), (tag, k)
        rc, rs = oracle.mx_encode_f32(ref.w)
        gc, gs = self.codes.view.cpu().numpy(), self.scales.view.cpu().numpy()
        if same:
            assert np.array_equal(gs, rs), (tag, np.nonzero(gs != rs)[0][:5])
            assert np.array_equal(gc, rc), (tag, np.nonzero(gc != rc)[0][:5])
        assert np.array_equal(st["p"], self.p_before), tag  # bf16 parameters untouched
        assert self.codes.intact() and self.scales.intact() and self.guards_intact(), tag


@pytest.mark.parametrize("n", [1, 31, 32, 33, 1000, 65_549, (1 << 20) + 40])
@pytest.mark.parametrize("p", [1, 8])
def test_mx_params_match_oracle(n, p):
    w0 = (np.random.default_rng(n + p).standard_normal(n) * 0.02).astype(np.float32)
    run = MxRun(w0, p)
    ref = oracle.OracleOptimizer(w0)
    for k, host in enumerate(edge_sequence(n, p, seed=n * 3 + p), start=1):
        zb.zg_step(run.ctx, [to_dev_bf16(h) for h in host], L)
        dec = ref.step(host, L)
        run.check(f"mx-params n={n} p={p} step {k}", ref, dec, zb.zg_get_info(run.ctx))


def test_mx_params_with_staged_variant_and_mx_gradients():
    n, p = 200_003, 8
    w0 = (np.random.default_rng(9).standard_normal(n) * 0.02).astype(np.float32)
    staged, mxwire = MxRun(w0, p, "staged"), MxRun(w0, p)
    ref_b, ref_m = oracle.OracleOptimizer(w0), oracle.OracleOptimizer(w0)
    for k in range(3):
        host = [synth.random_bf16(n, seed=40 + 10 * k + r, scale=(1e-3 if k != 1 else 1.0) * L) for r in range(p)]
        zb.zg_step(staged.ctx, [to_dev_bf16(h) for h in host], L)
        staged.check(f"staged step {k}", ref_b, ref_b.step(host, L), zb.zg_get_info(staged.ctx))
        enc = [oracle.mx_encode(h) for h in host]
        zb.zg_step_mxfp8(mxwire.ctx, [torch.from_numpy(c).cuda() for c, _ in enc],
                         [torch.from_numpy(s).cuda() for _, s in enc], L)
        dec = ref_m.step_mx([c for c, _ in enc], [s for _, s in enc], L)
        mxwire.check(f"mx wire step {k}", ref_m, dec, zb.zg_get_info(mxwire.ctx))


def test_mx_params_binding_rules():
    n, p = 4096, 2
    run = GpuRun(np.zeros(n, np.float32), p)
    codes = torch.zeros(n, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(n // 32, dtype=torch.uint8, device="cuda")
    lib = zb.lib()
    assert lib.zg_bind_params_mxfp8(run.ctx.handle, codes.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_bind_params_mxfp8(run.ctx.handle, codes.data_ptr() + 4, scales.data_ptr()) == zb.ZG_ERR_MISALIGNED
    zb.zg_bind_params_mxfp8(run.ctx, codes, scales)
    with pytest.raises(zb.ZgError):
        zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_TMA)
    # back to bf16 parameters
    zb.zg_bind_params_mxfp8(run.ctx, None, None)
    host = [synth.random_bf16(n, seed=r, scale=L) for r in range(p)]
    zb.zg_step(run.ctx, [to_dev_bf16(h) for h in host], L)
    assert zb.zg_get_info(run.ctx).step_t == 1
    w = to_host_f32(run.bufs["w"].view)
    pb = to_host_u16(run.bufs["p"].view)
    want = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(pb, want)
    assert not codes.any()  # MX buffers no longer written
