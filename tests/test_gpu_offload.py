"""Optimizer state moved off the card (Zero From Scratch, item 11): fp32 w, m,
v in pinned host memory, read and written in place by the same kernels over
the host link. Results must be the same bits as with the state in HBM."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import compare_state, to_dev_bf16, to_host_u16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu


def _state(opt):
    torch.cuda.synchronize()
    return {"w": opt.w.numpy().copy(), "m": opt.m.numpy().copy(), "v": opt.v.numpy().copy(),
            "p": to_host_u16(opt.params)}


@pytest.mark.parametrize("n,p", [(65_549, 4), (1 << 22, 8)])
def test_offloaded_state_matches_oracle(n, p):
    w0 = (np.random.default_rng(n).standard_normal(n) * 0.02).astype(np.float32)
    opt = zb.ShardedAdamW(n, p, zb.Hparams(), torch.from_numpy(w0), offload=True)
    assert not opt.w.is_cuda and opt.w.is_pinned() and opt.params.is_cuda
    ref = oracle.OracleOptimizer(w0)
    for k in range(3):
        host = [synth.random_bf16(n, seed=300 + 10 * k + r, scale=(1e-3 if k != 1 else 1.0) * 1024.0)
                for r in range(p)]
        opt.step([to_dev_bf16(h) for h in host], 1024.0)
        info = opt.info()
        dec = ref.step(host, 1024.0)
        assert info.status == 0 and info.found_inf == dec.found_inf and info.step_t == ref.t
        st = compare_state(f"offload n={n} p={p}/step{k + 1}", _state(opt),
                           {"w": ref.w, "m": ref.m, "v": ref.v, "p": ref.p}, 2e-6 * (k + 1))
        if info.clip_coef == dec.clip:
            assert st["w_bitexact"] == st["m_bitexact"] == st["v_bitexact"] == st["p_bitexact"] == 1.0


def test_offloaded_mx_step_matches_resident():
    n, p = 100_003, 8
    w0 = torch.from_numpy((np.random.default_rng(1).standard_normal(n) * 0.02).astype(np.float32))
    off = zb.ShardedAdamW(n, p, zb.Hparams(), w0, offload=True)
    res = zb.ShardedAdamW(n, p, zb.Hparams(), w0)
    for k in range(2):
        enc = [oracle.mx_encode(synth.random_bf16(n, seed=50 + 10 * k + r, scale=1e-3, dist="student_t"))
               for r in range(p)]
        codes = [torch.from_numpy(c).cuda() for c, _ in enc]
        scales = [torch.from_numpy(s).cuda() for _, s in enc]
        off.step_mxfp8(codes, scales, 1.0)
        res.step_mxfp8(codes, scales, 1.0)
    torch.cuda.synchronize()
    assert off.info().step_t == res.info().step_t == 2
    for a, b in ((off.w, res.w), (off.m, res.m), (off.v, res.v)):
        assert a.numpy().tobytes() == b.cpu().numpy().tobytes()
    assert torch.equal(off.params.view(torch.int16), res.params.view(torch.int16))
