"""Seeded random combinations of everything a step can be configured with,
each run on the GPU through the C ABI and on the oracle with the same bytes.

Per case the seed draws: N (log-uniform up to 4e5, so single elements,
ragged tails and multi-wave grids all occur), P in 1..16, the bf16 variant
(plain loads, TMA-staged, staged gradient), bf16 or MXFP8 gradients (encoded
on the GPU by zg_quant_mxfp8, checked against the oracle's encoding),
bf16 or MXFP8 stored parameters, averaging or plain sum, a power-of-two
loss scale, and the AdamW and clip settings (clip off, loose or tight).
Three steps run per case with fresh gradients of a random size; some cases
plant an inf or a NaN in the second step, which both sides must skip.

The bar is the one every parity test states: found-inf decisions and the
step count equal, the norm within 1e-5, w, m and v within 2e-6 per applied
step, bf16 parameters within one ulp, MX codes and scale bytes exact, and all
of it bit for bit whenever both sides took the same clip factor. Guard bytes
around the state buffers must stay untouched."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, log, to_dev_bf16, to_host_u16
from test_gpu_step import GpuRun, check_step
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = 200
STEPS = 3


def draw(seed: int) -> dict:
    rng = np.random.default_rng(0x5EED00 + seed)
    variant = str(rng.choice(["ldg", "tma", "staged"]))
    hp = dict(lr=float(10 ** rng.uniform(-4, -2)), beta1=float(rng.choice([0.9, 0.8])),
              beta2=float(rng.choice([0.999, 0.95])), eps=float(rng.choice([1e-8, 1e-6])),
              weight_decay=float(rng.choice([0.0, 0.01, 0.1])), max_grad_norm=float(rng.choice([0.0, 0.5, 1.0, 4.0])),
              norm_eps=1e-6, grad_average=int(rng.integers(0, 2)))
    return {
        "n": int(round(np.exp(rng.uniform(0, np.log(4e5))))),
        "p": int(rng.integers(1, 17)),
        "variant": variant,
        "mx_grads": bool(rng.integers(0, 2)),
        # the TMA variant writes bf16 parameters only
        "mx_params": variant != "tma" and bool(rng.integers(0, 2)),
        "loss_scale": float(2.0 ** int(rng.integers(0, 17))),
        "hp": hp,
        "sigmas": [float(rng.choice([1e-4, 1e-3, 3e-2])) for _ in range(STEPS)],
        "plant": str(rng.choice(["none", "none", "inf", "nan"])),
        "plant_at": float(rng.uniform()),
    }


def case_id(seed: int) -> str:
    c = draw(seed)
    return (f"{seed}-n{c['n']}-p{c['p']}-{c['variant']}{'-mxg' if c['mx_grads'] else ''}"
            f"{'-mxp' if c['mx_params'] else ''}")


@pytest.mark.parametrize("seed", range(CASES), ids=case_id)
def test_random_combination_matches_oracle(seed):
    c = draw(seed)
    n, p, L = c["n"], c["p"], c["loss_scale"]
    w0 = (np.random.default_rng(seed).standard_normal(n) * 0.02).astype(np.float32)
    run = GpuRun(w0, p, zb.Hparams(**c["hp"]))
    ref = oracle.OracleOptimizer(w0, oracle.Hparams(**c["hp"]))
    if c["variant"] == "staged":
        stage = torch.zeros(n, dtype=torch.float32, device="cuda")
        zb.zg_bind_grad_stage(run.ctx, stage)
        zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_STAGED)
    elif c["variant"] == "tma":
        zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_TMA)
    if c["mx_params"]:
        pcodes, pscales = Guarded(n, torch.uint8), Guarded((n + 31) // 32, torch.uint8)
        zb.zg_bind_params_mxfp8(run.ctx, pcodes.view, pscales.view)
        p_before = to_host_u16(run.bufs["p"].view).copy()

    for k in range(STEPS):
        host = [synth.random_bf16(n, seed=90_000 + 1000 * seed + 10 * k + r, scale=c["sigmas"][k] * L,
                                  dist="student_t" if c["mx_grads"] else "normal") for r in range(p)]
        if k == 1 and c["plant"] != "none":
            host[int(c["plant_at"] * p)][int(c["plant_at"] * n)] = 0x7F80 if c["plant"] == "inf" else 0xFFC1
        if c["mx_grads"]:
            codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(p)]
            scales = [torch.empty((n + 31) // 32, dtype=torch.uint8, device="cuda") for _ in range(p)]
            for r in range(p):
                zb.zg_quant_mxfp8(to_dev_bf16(host[r]), codes[r], scales[r], n)
            enc = [oracle.mx_encode(h) for h in host]
            for r in range(p):
                assert np.array_equal(codes[r].cpu().numpy(), enc[r][0]), (seed, k, r, "codes")
                assert np.array_equal(scales[r].cpu().numpy(), enc[r][1]), (seed, k, r, "scales")
            zb.zg_step_mxfp8(run.ctx, codes, scales, L)
            dec = ref.step_mx([e[0] for e in enc], [e[1] for e in enc], L)
        else:
            zb.zg_step(run.ctx, [to_dev_bf16(h) for h in host], L)
            dec = ref.step(host, L)
        info = zb.zg_get_info(run.ctx)
        if c["plant"] != "none" and k == 1:
            assert dec.found_inf and info.found_inf, (seed, info)
        if c["mx_params"]:
            # the bf16 buffer is left alone; the state is compared as usual and
            # the parameters as the oracle's encoding of its master weights
            assert np.array_equal(to_host_u16(run.bufs["p"].view), p_before), seed
            ref_p, ref.p = ref.p, p_before
            check_step(case_id(seed), run, ref, dec, info, k + 1)
            ref.p = ref_p
            if info.clip_coef == dec.clip:
                rc, rs = oracle.mx_encode_f32(ref.w)
                assert np.array_equal(pcodes.view.cpu().numpy(), rc), (seed, k, "param codes")
                assert np.array_equal(pscales.view.cpu().numpy(), rs), (seed, k, "param scales")
            assert pcodes.intact() and pscales.intact(), seed
        else:
            check_step(case_id(seed), run, ref, dec, info, k + 1)
        assert run.guards_intact(), seed
    log({"case": "random-combo", "seed": seed, **{k: v for k, v in c.items() if k != "hp"}, **c["hp"],
         "t": ref.t})


BUCKET_CASES = 60


def draw_buckets(seed: int) -> dict:
    """N, P, variant and a random partition of [0, N) into contiguous buckets
    whose inner edges are multiples of 8 (the bucket entry point's rule)."""
    rng = np.random.default_rng(0xB0C4E7 + seed)
    n = int(round(np.exp(rng.uniform(0, np.log(3e5)))))
    inner = np.arange(8, n, 8)
    k = int(min(inner.size, rng.integers(0, 12)))
    cuts = sorted(rng.choice(inner, size=k, replace=False).tolist()) if k else []
    edges = [0] + cuts + [n]
    return {"n": n, "p": int(rng.integers(1, 17)), "variant": str(rng.choice(["ldg", "tma", "staged"])),
            "buckets": list(zip(edges[:-1], edges[1:])), "plant": bool(rng.integers(0, 4) == 0),
            "plant_at": float(rng.uniform())}


@pytest.mark.parametrize("seed", range(BUCKET_CASES),
                         ids=lambda s: f"{s}-n{draw_buckets(s)['n']}-b{len(draw_buckets(s)['buckets'])}")
def test_random_bucket_partition_matches_oracle(seed):
    """The norm taken over a random bucket partition equals the whole-vector
    norm (same squares, fp64 sums associated per bucket: 1e-12), and the step
    that follows matches the oracle."""
    c = draw_buckets(seed)
    n, p, L = c["n"], c["p"], 1024.0
    w0 = (np.random.default_rng(seed + 77).standard_normal(n) * 0.02).astype(np.float32)
    run, whole = GpuRun(w0, p), GpuRun(w0, p)
    ref = oracle.OracleOptimizer(w0)
    if c["variant"] == "staged":
        stage = torch.zeros(n, dtype=torch.float32, device="cuda")
        zb.zg_bind_grad_stage(run.ctx, stage)
        zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_STAGED)
    elif c["variant"] == "tma":
        zb.zg_set_variant(run.ctx, zb.ZG_VARIANT_TMA)
    for k in range(STEPS):
        host = [synth.random_bf16(n, seed=190_000 + 1000 * seed + 10 * k + r, scale=(1e-3 if k != 1 else 0.3) * L)
                for r in range(p)]
        if k == 2 and c["plant"]:
            host[int(c["plant_at"] * p)][int(c["plant_at"] * n)] = 0x7F80
        dev = [to_dev_bf16(h) for h in host]
        last = len(c["buckets"]) - 1
        for i, (lo, hi) in enumerate(c["buckets"]):
            flags = (zb.ZG_BUCKET_FIRST if i == 0 else 0) | (zb.ZG_BUCKET_LAST if i == last else 0)
            zb.zg_grad_norm_bucket(run.ctx, dev, lo, hi, L, flags)
        zb.zg_grad_norm(whole.ctx, dev, L)
        a, b = zb.zg_get_info(run.ctx), zb.zg_get_info(whole.ctx)
        assert a.found_inf == b.found_inf, (seed, k)
        if not b.found_inf:
            assert abs(a.sumsq - b.sumsq) <= 1e-12 * b.sumsq, (seed, k, a.sumsq, b.sumsq)
        zb.zg_shard_step(run.ctx, dev, L)
        zb.zg_shard_step(whole.ctx, dev, L)
        dec = ref.step(host, L)
        check_step(f"random buckets {seed}", run, ref, dec, zb.zg_get_info(run.ctx), k + 1)
        assert run.guards_intact(), seed
