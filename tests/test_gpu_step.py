"""GPU step vs the oracle on small, ragged and degenerate cases, through the C ABI.

Each case runs a sequence of steps on the same seeded bf16 inputs on both
sides: an ordinary step, a step whose norm triggers the clip, a step with
+inf on one rank and one with NaN on another (both must be skipped), then an
ordinary step again. The GPU result must match the oracle within the stated
tolerances (w, m, v relative 2e-6 per step; bf16 params 1 ulp; norm 1e-5;
skip decisions exactly), and bit for bit whenever both sides chose the same
clip factor, since both run the same correctly rounded fp32 sequence. Guard
canaries around every state buffer catch writes outside [0, N).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, compare_state, log, to_dev_bf16, to_host_f32, to_host_u16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

L = 1024.0


class GpuRun:
    """A context over guarded state buffers, initialised from w0."""

    def __init__(self, w0: np.ndarray, p: int, hp=zb.Hparams()):
        n = w0.size
        self.n, self.p = n, p
        self.ctx = zb.zg_init(n, p, hp)
        self.bufs = {k: Guarded(n, torch.float32) for k in ("w", "m", "v")}
        self.bufs["p"] = Guarded(n, torch.bfloat16)
        self.bufs["w"].view.copy_(torch.from_numpy(w0))
        self.bufs["m"].view.zero_()
        self.bufs["v"].view.zero_()
        self.bufs["p"].view.zero_()
        zb.zg_bind(self.ctx, *(self.bufs[k].view for k in ("w", "m", "v", "p")))

    def state(self) -> dict:
        return {"w": to_host_f32(self.bufs["w"].view), "m": to_host_f32(self.bufs["m"].view),
                "v": to_host_f32(self.bufs["v"].view), "p": to_host_u16(self.bufs["p"].view)}

    def guards_intact(self) -> bool:
        return all(b.intact() for b in self.bufs.values())


def ref_state(ref: oracle.OracleOptimizer) -> dict:
    return {"w": ref.w, "m": ref.m, "v": ref.v, "p": ref.p}


def check_step(tag, run: GpuRun, ref, dec, info, step_no):
    assert info.status == 0, (tag, info)
    assert info.found_inf == dec.found_inf, (tag, info, dec)
    assert info.step_t == ref.t, (tag, info.step_t, ref.t)
    if not dec.found_inf:
        assert abs(info.norm - dec.norm) <= 1e-5 * dec.norm + 1e-300, (tag, info.norm, dec.norm)
    st = compare_state(f"{tag}/step{step_no}", run.state(), ref_state(ref), min(1e-5, 2e-6 * max(ref.t, 1)))
    if info.clip_coef == dec.clip:
        for k in ("w", "m", "v", "p"):
            assert st[f"{k}_bitexact"] == 1.0, (tag, k, st)
    return st


def edge_sequence(n: int, p: int, seed: int):
    """Five steps of P bf16 buffers: ordinary, large (clips), +inf at index 0
    of the last rank, NaN at the last index of rank 0, ordinary."""
    steps = []
    for k, scale in enumerate((1e-3, 1.0, 1e-3, 1e-3, 1e-3)):
        bufs = [synth.random_bf16(n, seed=seed * 1000 + 10 * k + r, scale=scale * L) for r in range(p)]
        if k == 2:
            bufs[p - 1][0] = 0x7F80
        if k == 3:
            bufs[0][n - 1] = 0x7FC0
        steps.append(bufs)
    return steps


@pytest.mark.parametrize("n", [1, 7, 8, 31, 32, 33, 1000, 65_549])
@pytest.mark.parametrize("p", [1, 2, 3, 4, 8, 16])
def test_edge_shapes(n, p):
    rng = np.random.default_rng(n * 31 + p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p)
    ref = oracle.OracleOptimizer(w0)
    saw_clip = False
    for k, host in enumerate(edge_sequence(n, p, seed=n * 17 + p), start=1):
        dev = [Guarded(n, torch.bfloat16) for _ in range(p)]
        for r in range(p):
            to_dev_bf16(host[r], dev[r].view)
        zb.zg_step(run.ctx, [d.view for d in dev], L)
        info = zb.zg_get_info(run.ctx)
        dec = ref.step(host, L)
        saw_clip |= (not dec.found_inf and dec.clip < 1.0)
        check_step(f"edge n={n} p={p}", run, ref, dec, info, k)
        assert all(d.intact() for d in dev)
    assert run.guards_intact()
    assert ref.t == 3
    if n >= 64:
        assert saw_clip


def _small_case(n=4099, p=4, steps=4, seed=3):
    rng = np.random.default_rng(seed)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    host = [[synth.random_bf16(n, seed=seed * 100 + 10 * t + r, scale=0.05 * L) for r in range(p)]
            for t in range(steps)]
    return w0, host


def test_repeat_is_bit_identical():
    w0, host = _small_case()
    outs = []
    for _ in range(2):
        run = GpuRun(w0, 4)
        norms = []
        for h in host:
            zb.zg_step(run.ctx, [to_dev_bf16(x) for x in h], L)
            norms.append(zb.zg_get_info(run.ctx).sumsq)
        s = run.state()
        outs.append((norms, {k: s[k].tobytes() for k in s}))
    assert outs[0] == outs[1]


def test_stale_norm_is_refused_and_writes_nothing():
    w0, host = _small_case(steps=1)
    run = GpuRun(w0, 4)
    dev = [to_dev_bf16(x) for x in host[0]]
    zb.zg_grad_norm(run.ctx, dev, L)
    zb.zg_shard_step(run.ctx, dev, L)
    after_one = run.state()
    assert zb.zg_get_info(run.ctx).status == 0
    zb.zg_shard_step(run.ctx, dev, L)  # no fresh norm
    info = zb.zg_get_info(run.ctx)
    assert info.status == zb.ZG_ERR_STALE_NORM and info.step_t == 1
    again = run.state()
    for k in after_one:
        assert after_one[k].tobytes() == again[k].tobytes()
    assert zb.zg_get_info(run.ctx).status == 0  # the status was cleared by the read


def test_resume_matches_uninterrupted():
    w0, host = _small_case(steps=6)
    full = GpuRun(w0, 4)
    for h in host:
        zb.zg_step(full.ctx, [to_dev_bf16(x) for x in h], L)
    first = GpuRun(w0, 4)
    for h in host[:3]:
        zb.zg_step(first.ctx, [to_dev_bf16(x) for x in h], L)
    saved = first.state()
    t = zb.zg_get_info(first.ctx).step_t
    resumed = GpuRun(saved["w"], 4)
    resumed.bufs["m"].view.copy_(torch.from_numpy(saved["m"]))
    resumed.bufs["v"].view.copy_(torch.from_numpy(saved["v"]))
    zb.zg_set_step(resumed.ctx, t)
    for h in host[3:]:
        zb.zg_step(resumed.ctx, [to_dev_bf16(x) for x in h], L)
    a, b = full.state(), resumed.state()
    for k in a:
        assert a[k].tobytes() == b[k].tobytes(), k
    assert zb.zg_get_info(resumed.ctx).step_t == 6


def test_resume_is_stream_ordered_and_waits_for_no_other_stream():
    """zg_set_step is queued on the stream it is given: it returns while
    another stream is still busy (a long chain of copies), and takes effect
    in order on its own stream, so the next step there counts from t."""
    w0, host = _small_case(steps=1)
    run = GpuRun(w0, 4)
    ref = GpuRun(w0, 4)
    dev = [to_dev_bf16(x) for x in host[0]]
    src = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    busy, mine = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(200):  # tens of milliseconds of copying on another stream
        zb.zg_probe_copy(src, dst, busy)
    zb.zg_set_step(run.ctx, 5, mine)
    zb.zg_step(run.ctx, dev, L, stream=mine)
    assert not busy.query()  # neither call waited for the busy stream
    info = zb.zg_get_info(run.ctx, mine)
    assert info.status == 0 and info.step_t == 6
    busy.synchronize()
    # the same as resuming an idle context the same way
    zb.zg_set_step(ref.ctx, 5)
    zb.zg_step(ref.ctx, dev, L)
    a, b = run.state(), ref.state()
    for k in a:
        assert a[k].tobytes() == b[k].tobytes(), k


def test_loss_scale_invariance_on_gpu():
    n, p = 3001, 3
    rng = np.random.default_rng(8)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    base = [synth.random_bf16(n, seed=40 + r, scale=1e-3) for r in range(p)]
    res = []
    for ls in (1024.0, 65536.0):
        scaled = [(oracle.bf16_to_f32(b) * np.float32(ls)).view(np.uint32) >> 16 for b in base]
        run = GpuRun(w0, p)
        for _ in range(3):
            zb.zg_step(run.ctx, [to_dev_bf16(s.astype(np.uint16)) for s in scaled], ls)
        res.append({k: v.tobytes() for k, v in run.state().items()})
    assert res[0] == res[1]


def test_side_stream_and_two_contexts():
    w0, host = _small_case(steps=2)
    ref = oracle.OracleOptimizer(w0)
    runs = [GpuRun(w0, 4), GpuRun(w0, 4)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for h in host:
            dev = [to_dev_bf16(x) for x in h]
            for run in runs:
                zb.zg_step(run.ctx, dev, L, stream=s)
    s.synchronize()
    for h in host:
        ref.step(h, L)
    for run in runs:
        st = compare_state("side-stream", run.state(), ref_state(ref), 4e-6)
        assert st["w_bitexact"] == 1.0 or zb.zg_get_info(run.ctx, s).clip_coef != 1.0


def test_sum_without_average_and_clip_off():
    n, p = 2049, 2
    rng = np.random.default_rng(5)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp_b = zb.Hparams(max_grad_norm=0.0, grad_average=0, weight_decay=0.0)
    hp_o = oracle.Hparams(max_grad_norm=0.0, grad_average=0, weight_decay=0.0)
    run = GpuRun(w0, p, hp_b)
    ref = oracle.OracleOptimizer(w0, hp_o)
    for t in range(3):
        host = [synth.random_bf16(n, seed=70 + 10 * t + r, scale=3.0 * L) for r in range(p)]
        zb.zg_step(run.ctx, [to_dev_bf16(x) for x in host], L)
        dec = ref.step(host, L)
        info = zb.zg_get_info(run.ctx)
        assert info.clip_coef == 1.0 and dec.clip == 1.0
        check_step("sum-no-clip", run, ref, dec, info, t + 1)


def test_argument_errors():
    n, p = 64, 2
    ctx = zb.zg_init(n, p)
    dev = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    with pytest.raises(zb.ZgError) as e:
        zb.zg_step(ctx, dev, L)
    assert e.value.code == zb.ZG_ERR_NOT_BOUND
    st = [torch.zeros(n + 8, dtype=torch.float32, device="cuda") for _ in range(3)]
    params = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    lib = zb.lib()
    rc = lib.zg_bind(ctx.handle, st[0].data_ptr() + 4, st[1].data_ptr(), st[2].data_ptr(), params.data_ptr())
    assert rc == zb.ZG_ERR_MISALIGNED
    zb.zg_bind(ctx, st[0], st[1], st[2], params)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(zb.ZgError) as e:
            zb.zg_step(ctx, dev, bad)
        assert e.value.code == zb.ZG_ERR_INVALID_ARG
    ptrs = (zb.ctypes.c_void_p * 2)(dev[0].data_ptr(), dev[1].data_ptr() + 2)
    assert lib.zg_step(ctx.handle, ptrs, L, None) == zb.ZG_ERR_MISALIGNED
    ptrs = (zb.ctypes.c_void_p * 2)(dev[0].data_ptr(), None)
    assert lib.zg_step(ctx.handle, ptrs, L, None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_set_variant(ctx.handle, 7) == zb.ZG_ERR_INVALID_ARG
    assert zb.zg_get_info(ctx).step_t == 0  # nothing ran
    log({"case": "argument-errors", "ok": True})


@pytest.mark.parametrize("path", ["ldg", "tma", "staged", "mx", "mx_staged"])
def test_repeat_is_bit_identical_every_path(path):
    """Same inputs twice through each kernel path, at a size that fills every
    SM with several blocks: the norm (fixed grid, fixed partial order) and
    every state byte must repeat exactly."""
    n, p = (1 << 22) + 13, 8
    rng = np.random.default_rng(17)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    host = [[synth.random_bf16(n, seed=900 + 10 * t + r, scale=(1e-3 if t != 1 else 1.0) * L,
                               dist="student_t") for r in range(p)] for t in range(3)]
    mx = path.startswith("mx")
    if mx:
        enc = [[oracle.mx_encode(h) for h in step] for step in host]
    outs = []
    for _ in range(2):
        run = GpuRun(w0, p)
        if path in ("staged", "mx_staged"):
            stage = torch.zeros(n, dtype=torch.float32, device="cuda")
            zb.zg_bind_grad_stage(run.ctx, stage)
            zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_STAGED)
        elif path == "tma":
            zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_TMA)
        sums = []
        for t in range(3):
            if mx:
                zb.zg_step_mxfp8(run.ctx, [torch.from_numpy(c).cuda() for c, _ in enc[t]],
                                 [torch.from_numpy(s).cuda() for _, s in enc[t]], L)
            else:
                zb.zg_step(run.ctx, [to_dev_bf16(x) for x in host[t]], L)
            info = zb.zg_get_info(run.ctx)
            assert info.status == 0 and not info.found_inf, (path, t, info)
            sums.append(info.sumsq)
        s = run.state()
        outs.append((sums, {k: s[k].tobytes() for k in s}))
        assert run.guards_intact()
    assert outs[0] == outs[1], path
