"""The MXFP8 path on the GPU vs the oracle: codes and scale bytes bit-exact,
and the step from decoded codes within the step tolerances
(Zero From Scratch, item 14: E4M3 elements, one power-of-two scale per 32)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, log, to_dev_bf16
from test_gpu_step import GpuRun, check_step
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu


def gpu_encode(x: np.ndarray):
    n = x.size
    codes = Guarded(n, torch.uint8)
    scales = Guarded((n + 31) // 32, torch.uint8)
    zb.zg_quant_mxfp8(to_dev_bf16(x), codes.view, scales.view, n)
    torch.cuda.synchronize()
    assert codes.intact() and scales.intact()
    return codes.view.cpu().numpy(), scales.view.cpu().numpy()


def special_blocks() -> np.ndarray:
    """Hand-made blocks: zeros and negative zeros, bf16 subnormals, amax at
    448 * 2^k and just below 512 * 2^k, ties between E4M3 neighbours, huge
    and tiny magnitudes, and blocks poisoned by inf or NaN."""
    f = lambda vals: (np.array(vals, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    blocks = [np.zeros(32, np.uint16), np.full(32, 0x8000, np.uint16), np.arange(32, dtype=np.uint16)]
    for k in (-130, -20, 0, 7, 100, 119):
        b = np.zeros(32, np.float32)
        b[0] = 448.0 * 2.0 ** k if k > -126 else 2.0 ** -126
        b[1:] = np.linspace(-1, 1, 31) * 2.0 ** k
        blocks.append(f(b))
        blocks.append(f(np.full(32, 510.0 * 2.0 ** min(k, 119))))
    tie = np.zeros(32, np.float32)
    tie[0] = 1.0
    tie[1:9] = [2.0 ** -17, 2.0 ** -18, 3 * 2.0 ** -19, -(2.0 ** -20), 1.0625, 1.1875, -1.0625, 17.0 / 16]
    blocks.append(f(tie))
    for bad in (0x7F80, 0xFF80, 0x7FC0, 0xFFC1):
        b = f(np.linspace(-3, 3, 32))
        b[13] = bad
        blocks.append(b)
    return np.concatenate(blocks)


@pytest.mark.parametrize("tail", [0, 1, 8, 13, 31])
def test_quant_bit_exact(tail):
    parts = [special_blocks(),
             np.arange(65536, dtype=np.uint32).astype(np.uint16),  # every bf16 pattern
             np.random.default_rng(2).permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16)),
             synth.random_bf16(32 * 4000, seed=1, scale=1e-3, dist="student_t"),
             synth.random_bf16(32 * 4000, seed=2, scale=1.0, dist="logspread")]
    x = np.concatenate(parts)
    x = x[: (x.size // 32) * 32 - (32 - tail) % 32] if tail else x[: (x.size // 32) * 32]
    gc, gs = gpu_encode(x)
    rc, rs = oracle.mx_encode(x)
    bad_c = np.nonzero(gc != rc)[0]
    bad_s = np.nonzero(gs != rs)[0]
    log({"case": f"mx-quant tail={tail}", "n": int(x.size), "code_mismatch": int(bad_c.size),
         "scale_mismatch": int(bad_s.size)})
    assert bad_s.size == 0, [(int(i), int(gs[i]), int(rs[i])) for i in bad_s[:8]]
    assert bad_c.size == 0, [(int(i), hex(x[i]), int(gc[i]), int(rc[i])) for i in bad_c[:8]]


def test_quant_empty_and_tiny():
    for n in (1, 2, 31, 33):
        x = synth.random_bf16(n, seed=n, scale=3.0)
        gc, gs = gpu_encode(x)
        rc, rs = oracle.mx_encode(x)
        assert np.array_equal(gc, rc) and np.array_equal(gs, rs)
    zb.zg_quant_mxfp8(torch.zeros(8, dtype=torch.bfloat16, device="cuda"),
                      torch.zeros(8, dtype=torch.uint8, device="cuda"),
                      torch.zeros(1, dtype=torch.uint8, device="cuda"), n=0)


@pytest.mark.parametrize("n,p", [(1, 1), (33, 2), (1000, 3), (30_001, 5), (65_549, 8), (20_011, 11), (4096, 16)])
def test_mx_step_small(n, p):
    rng = np.random.default_rng(n + p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p)
    ref = oracle.OracleOptimizer(w0)
    for k in range(4):
        host = [synth.random_bf16(n, seed=500 + 10 * k + r, scale=1e-3 if k != 1 else 1.0, dist="student_t")
                for r in range(p)]
        if k == 2:
            host[p - 1][n - 1] = 0x7F80
        enc = [oracle.mx_encode(h) for h in host]
        codes = [torch.from_numpy(c).cuda() for c, _ in enc]
        scales = [torch.from_numpy(s).cuda() for _, s in enc]
        zb.zg_step_mxfp8(run.ctx, codes, scales, 1.0)
        info = zb.zg_get_info(run.ctx)
        dec = ref.step_mx([c for c, _ in enc], [s for _, s in enc], 1.0)
        check_step(f"mx-step n={n} p={p}", run, ref, dec, info, k + 1)
    assert ref.t == 3


def test_mx_step_raw_bytes():
    """MX inputs as raw bytes rather than encoder output: random codes at
    scales from subnormal (0) to large, blocks whose scale bytes (247..254)
    the encoder never writes, a block whose products overflow and a NaN
    code. Both ways the GPU sums decoded products (fused packed multiply-add
    for ordinary scales, separate multiply and add otherwise) must match the
    oracle, skips included."""
    n, p = 65_549, 4
    nb = (n + 31) // 32
    rng = np.random.default_rng(77)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p)
    ref = oracle.OracleOptimizer(w0)
    big_blocks = rng.choice(nb, 40, replace=False)
    for k in range(5):
        codes, scales = [], []
        for r in range(p):
            c = rng.integers(0, 256, n).astype(np.uint8)
            c[(c & 0x7F) == 0x7F] = 0x3A  # no NaN codes
            s = rng.integers(100, 136, nb).astype(np.uint8)
            s[rng.choice(nb, 30, replace=False)] = 0  # subnormal scale
            s[big_blocks] = rng.integers(247, 255, big_blocks.size)
            for b in big_blocks:  # those blocks hold zeros (finite products) ...
                c[32 * b:32 * b + 32] = 0
            codes.append(c)
            scales.append(s)
        if k == 2:  # ... except here: a product that overflows -> inf -> skip
            codes[1][32 * int(big_blocks[0]) + 5] = 0x40
        if k == 3:  # a NaN code -> skip
            codes[2][n // 2] = 0xFF
        zb.zg_step_mxfp8(run.ctx, [torch.from_numpy(c).cuda() for c in codes],
                         [torch.from_numpy(s).cuda() for s in scales], 1.0)
        info = zb.zg_get_info(run.ctx)
        dec = ref.step_mx(codes, scales, 1.0)
        assert bool(dec.found_inf) == (k in (2, 3)), (k, dec.found_inf)
        check_step(f"mx-raw step {k + 1}", run, ref, dec, info, k + 1)
    assert ref.t == 3


def _lossless_bf16(n: int, seed: int) -> np.ndarray:
    """bf16 values every one of which MXFP8 encodes exactly: per 32-block,
    +-(1 + k/8) 2^j with k <= 6 and j within six binades of the block's top
    exponent, which one value carries."""
    r = np.random.default_rng(seed)
    x = np.empty(n, np.float32)
    for b in range(0, n, 32):
        m = min(32, n - b)
        top = int(r.integers(-8, 4))
        d = r.integers(0, 7, m)
        d[0] = 0
        x[b:b + m] = r.choice([-1.0, 1.0], m) * (1 + r.integers(0, 7, m) / 8) * 2.0 ** (top - d)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("n,p", [(4099, 4), ((1 << 20) + 96, 8)])
def test_mx_step_on_lossless_gradients_equals_bf16_step(n, p):
    """Encoded on the GPU, gradients MXFP8 holds exactly must give the MX step
    the bf16 step's bits (the two decode paths meet on the same fp32 values).
    The two norm passes add the same squares in different orders (the bf16
    pass exactly over warp chunks, the MX pass over its own fixed grid), so
    their sums of squares agree to 1e-12; the clip factor (1 here) and the
    state must be the same bits."""
    w0 = (np.random.default_rng(n).standard_normal(n) * 0.02).astype(np.float32)
    a, b = GpuRun(w0, p), GpuRun(w0, p)
    for t in range(3):
        host = [_lossless_bf16(n, 1000 * t + r) for r in range(p)]
        dev = [to_dev_bf16(h) for h in host]
        codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(p)]
        scales = [torch.empty((n + 31) // 32, dtype=torch.uint8, device="cuda") for _ in range(p)]
        for r in range(p):
            zb.zg_quant_mxfp8(dev[r], codes[r], scales[r], n)
        zb.zg_step(a.ctx, dev, 1024.0)
        zb.zg_step_mxfp8(b.ctx, codes, scales, 1024.0)
        ia, ib = zb.zg_get_info(a.ctx), zb.zg_get_info(b.ctx)
        assert ia.status == ib.status == 0 and ia.clip_coef == ib.clip_coef == 1.0, (t, ia, ib)
        assert abs(ia.sumsq - ib.sumsq) <= 1e-12 * ib.sumsq, (t, ia, ib)
    sa, sb = a.state(), b.state()
    for k in sa:
        assert sa[k].tobytes() == sb[k].tobytes(), k


@pytest.mark.parametrize("n,p", [(1, 1), (7, 2), (4099, 4), (65_549, 8), ((1 << 20) + 13, 8), (300_017, 16)])
def test_quant_norm_equals_bf16_norm_on_lossless_gradients(n, p):
    """On gradients MXFP8 holds exactly, the fused encode-and-norm pass forms
    the bf16 norm pass's g (exact decoded products summed in rank order) and
    sums its squares the same way (the same warp chunks over g padded to
    whole vectors, the same butterfly, the same exact total): the same bits,
    ragged N included."""
    host = [_lossless_bf16(n, 77 * n + r) for r in range(p)]
    dev = [to_dev_bf16(h) for h in host]
    a, b = zb.zg_init(n, p), zb.zg_init(n, p)
    nb = (n + 31) // 32
    codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(p)]
    scales = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(p)]
    zb.zg_grad_norm(a, dev, 1024.0)
    zb.zg_quant_norm_mxfp8(b, dev, codes, scales, 1024.0)
    ia, ib = zb.zg_get_info(a), zb.zg_get_info(b)
    assert ia.status == ib.status == 0 and not ia.found_inf
    assert (ia.sumsq, ia.norm, ia.clip_coef) == (ib.sumsq, ib.norm, ib.clip_coef), (n, p, ia, ib)


@pytest.mark.parametrize("n,p", [(1, 1), (7, 2), (33, 3), (1000, 8), (65_549, 8), (20_011, 11), (4096, 16),
                                 (300_017, 4)])
@pytest.mark.parametrize("staged", [False, True])
def test_quant_norm_matches_encoder_separate_norm_and_oracle(n, p, staged):
    """zg_quant_norm_mxfp8 (every rank encoded and the norm taken in one pass)
    writes the encoder's codes and scale bytes bit for bit (the oracle's
    encoding), makes the separate MX norm pass's decision (the same skip and
    clip, the norm to 1e-12), and the step from its payload matches the
    oracle, bit for bit when the clip factors agree; a step with +inf and
    one with NaN are skipped. With the staged variant it also stores the
    reduced gradient the staged step reads."""
    rng = np.random.default_rng(n * 7 + p)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    fused, separate = GpuRun(w0, p), GpuRun(w0, p)
    if staged:
        for run in (fused, separate):
            run.stage = torch.empty(n, dtype=torch.float32, device="cuda")
            zb.zg_bind_grad_stage(run.ctx, run.stage)
            zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_STAGED)
    ref = oracle.OracleOptimizer(w0)
    nb = (n + 31) // 32
    for k in range(5):
        host = [synth.random_bf16(n, seed=800 + 10 * k + r, scale=1e-3 if k != 1 else 1.0, dist="student_t")
                for r in range(p)]
        if k == 2:
            host[p - 1][n - 1] = 0x7F80
        if k == 3:
            host[0][0] = 0x7FC0
        dev = [to_dev_bf16(h) for h in host]
        codes = [Guarded(n, torch.uint8) for _ in range(p)]
        scales = [Guarded(nb, torch.uint8) for _ in range(p)]
        zb.zg_quant_norm_mxfp8(fused.ctx, dev, [c.view for c in codes], [s.view for s in scales], 1.0)
        zb.zg_shard_step_mxfp8(fused.ctx, [c.view for c in codes], [s.view for s in scales], 1.0)
        info = zb.zg_get_info(fused.ctx)
        enc = [oracle.mx_encode(h) for h in host]
        for r in range(p):
            assert np.array_equal(codes[r].view.cpu().numpy(), enc[r][0]), (n, p, k, r, "codes")
            assert np.array_equal(scales[r].view.cpu().numpy(), enc[r][1]), (n, p, k, r, "scales")
            assert codes[r].intact() and scales[r].intact()
        c2 = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(p)]
        s2 = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(p)]
        for r in range(p):
            zb.zg_quant_mxfp8(dev[r], c2[r], s2[r], n)
        zb.zg_step_mxfp8(separate.ctx, c2, s2, 1.0)
        info2 = zb.zg_get_info(separate.ctx)
        assert info.found_inf == info2.found_inf == (k in (2, 3)), (k, info, info2)
        if not info.found_inf:
            assert abs(info.sumsq - info2.sumsq) <= 1e-12 * info2.sumsq, (k, info, info2)
        dec = ref.step_mx([c for c, _ in enc], [s for _, s in enc], 1.0)
        check_step(f"quant-norm n={n} p={p} staged={staged}", fused, ref, dec, info, k + 1)
        if info.clip_coef == info2.clip_coef:
            a, b = fused.state(), separate.state()
            for key in a:
                assert a[key].tobytes() == b[key].tobytes(), (n, p, k, key)
    assert ref.t == 3 and fused.guards_intact()
