"""Pins for the oracle: checks against facts that do not come from the oracle.

Each pin is a function of the loaded oracle library (a ctypes handle), so the
same pins run against the real oracle (``test_oracle_pins.py``) and against
copies with a planted mistake (``test_oracle_mutants.py``), which must fail at
least one of them.

What pins what:
  - first-step closed form: with m = v = 0 and t = 1 the bias-corrected
    update is lr * g / (|g| + eps) (the textbook AdamW reduces to it);
  - constant-gradient closed form: for a gradient held fixed, m_t = (1 -
    beta1^t) g and v_t = (1 - beta2^t) g^2, so every step moves w by
    lr * g / (|g| + eps);
  - weight decay closed form: w (1 - lr wd) - lr g / (|g| + eps);
  - two-step closed form with two different gradients, written out;
  - the clip + AdamW chain against torch.nn.utils.clip_grad_norm_ and
    torch.optim.AdamW (another rounding order, so to rounding);
  - the parameters after a step are the torch bf16 cast of the new weights;
  - clip: a vector of one repeated value has norm |a| sqrt(N);
  - norm: index-order binary64 sum vs math.fsum (correctly rounded);
  - averaging and loss scale on integer-valued gradients (exact);
  - skip: state bit-identical after a non-finite gradient;
  - bf16 rounding vs the torch cast; E4M3 values vs torch's float8_e4m3fn;
    the encoder vs a nearest-value table search with ties to even;
  - the MX scale rule on blocks built by hand from the format;
  - the MX round trip within half an E4M3 spacing at the block's scale;
  - shard layout invariants; identical learning (sharded == unsharded);
  - resume (set_step) reproduces an uninterrupted run;
  - power-of-two loss-scale invariance of the whole step;
  - stage three's gather: shards holding their own flat indices read back as
    the indices; MX shards built by hand from the formats and random ones
    decoded through torch's float8 values and bf16 cast.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

F32 = np.float32


def _ulp(x: float) -> float:
    return float(np.spacing(np.abs(F32(x))))


def _bf16(x) -> np.ndarray:
    """Exact bf16 patterns for values that are exactly representable."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def _trunc(x) -> np.ndarray:
    """bf16 patterns of float32 values truncated to bf16 (low half dropped):
    test inputs that are bf16 by construction."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _sp(x) -> np.ndarray:
    """binary32 spacing at |x|, as float64."""
    return np.spacing(np.abs(np.asarray(x, dtype=np.float64)).astype(np.float32)).astype(np.float64)


def _opt(lib, w0, **hp):
    return oracle.OracleOptimizer(np.asarray(w0, dtype=np.float32), oracle.Hparams(**hp), lib=lib)


# ------------------------------------------------------------- AdamW

def pin_first_step_closed_form(lib):
    gvals = np.array([1e-3, -2.5e-3, 3e-6, -7e-8, 1e-8, -1e-8, 0.75, -12.0, 4e-9, 0.0], dtype=np.float32)
    g = _trunc(gvals)
    gb = oracle.bf16_to_f32(g).astype(np.float64)
    lr, eps = 1e-3, 1e-8
    opt = _opt(lib, np.zeros(g.size), lr=lr, eps=eps, weight_decay=0.0, max_grad_norm=0.0)
    d = opt.step([g], 1.0)
    assert not d.found_inf and opt.t == 1
    expect = -lr * gb / (np.abs(gb) + eps)
    for got, want in zip(opt.w, expect):
        assert abs(float(got) - want) <= 2 * _ulp(want) + 1e-45, (got, want)
    # m and v after one step: (1 - beta) times g and g^2
    assert np.allclose(opt.m, 0.1 * gb, rtol=2e-7, atol=0)
    assert np.allclose(opt.v, 0.001 * gb * gb, rtol=4e-7, atol=1e-45)


def pin_first_step_weight_decay(lib):
    rng = np.random.default_rng(11)
    w0 = (rng.standard_normal(64) * 0.02).astype(np.float32)
    g = _trunc(rng.standard_normal(64).astype(np.float32) * F32(1e-3))
    gb = oracle.bf16_to_f32(g).astype(np.float64)
    lr, wd, eps = 1e-3, 0.01, 1e-8
    opt = _opt(lib, w0, lr=lr, weight_decay=wd, eps=eps, max_grad_norm=0.0)
    opt.step([g], 1.0)
    w0d = w0.astype(np.float64)
    dw = -lr * gb / (np.abs(gb) + eps)
    expect = w0d * (1.0 - lr * wd) + dw
    err = np.abs(opt.w.astype(np.float64) - expect)
    # a few roundings on operands of the size of w0 and of the update
    tol = 2 * (_sp(w0d) + _sp(dw) + _sp(expect))
    assert np.all(err <= tol), np.max(err / tol)


def pin_constant_gradient(lib):
    """Held gradient: bias correction makes every step the same size."""
    gvals = np.array([1e-3, -4e-4, 2.0, -3e-7, 5e-9], dtype=np.float32)
    g = _trunc(gvals)
    gb = oracle.bf16_to_f32(g).astype(np.float64)
    lr, eps, b1, b2 = 1e-3, 1e-8, 0.9, 0.999
    opt = _opt(lib, np.zeros(g.size), lr=lr, eps=eps, weight_decay=0.0, max_grad_norm=0.0)
    prev = opt.w.astype(np.float64).copy()
    for t in range(1, 31):
        opt.step([g], 1.0)
        assert opt.t == t
        dw = opt.w.astype(np.float64) - prev
        prev = opt.w.astype(np.float64).copy()
        want = -lr * gb / (np.abs(gb) + eps)
        assert np.all(np.abs(dw - want) <= 2e-5 * np.abs(want) + 1e-9 * lr), (t, dw, want)
        assert np.allclose(opt.m, (1 - b1 ** t) * gb, rtol=1e-5, atol=0)
        assert np.allclose(opt.v, (1 - b2 ** t) * gb * gb, rtol=1e-5, atol=1e-45)


def pin_two_step_closed_form(lib):
    rng = np.random.default_rng(5)
    n = 32
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g1 = _trunc(rng.standard_normal(n) * 1e-3)
    g2 = _trunc(rng.standard_normal(n) * 1e-3)
    a, b = oracle.bf16_to_f32(g1).astype(np.float64), oracle.bf16_to_f32(g2).astype(np.float64)
    lr, wd, eps, b1, b2 = 1e-3, 0.01, 1e-8, 0.9, 0.999
    opt = _opt(lib, w0, lr=lr, weight_decay=wd, eps=eps, max_grad_norm=0.0)
    opt.step([g1], 1.0)
    opt.step([g2], 1.0)
    w1 = w0.astype(np.float64) * (1 - lr * wd) - lr * a / (np.abs(a) + eps)
    m2 = b1 * (1 - b1) * a + (1 - b1) * b
    v2 = b2 * (1 - b2) * a * a + (1 - b2) * b * b
    mh, vh = m2 / (1 - b1 ** 2), v2 / (1 - b2 ** 2)
    dw2 = -lr * mh / (np.sqrt(vh) + eps)
    w2 = w1 * (1 - lr * wd) + dw2
    tol = 4 * (_sp(w0) + _sp(w1) + _sp(dw2) + _sp(w2))
    assert np.all(np.abs(opt.w - w2) <= tol), np.max(np.abs(opt.w - w2) / tol)
    assert np.allclose(opt.m, m2, rtol=1e-6)
    assert np.allclose(opt.v, v2, rtol=1e-6)


# ------------------------------------------------------------- clip and norm

def pin_adamw_and_clip_vs_torch(lib):
    """The whole clip + AdamW chain against PyTorch's own implementation of
    the same algorithm (torch.nn.utils.clip_grad_norm_, whose coefficient is
    max_norm / (norm + 1e-6) clamped to 1, then torch.optim.AdamW, single-tensor
    path): one rank, loss scale 1, so the oracle's gradient is the bf16 value
    itself. PyTorch rounds in another order (a lerp for m, sqrt(v) / sqrt(bc2)
    for the denominator, its norm in binary32), so the two agree to rounding,
    over steps that clip and steps that do not; a wrong beta, sign, bias
    correction, eps placement, clip rule or decay form shows as a large error."""
    import torch

    rng = np.random.default_rng(20)
    n = 4096
    hp = oracle.Hparams()
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    ref = _opt(lib, w0)
    param = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    topt = torch.optim.AdamW([param], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                             weight_decay=hp.weight_decay, foreach=False)
    clipped = unclipped = 0
    for t, sigma in enumerate((1e-3, 0.05, 2e-3, 0.1, 1e-3, 0.03)):
        g = _trunc(rng.standard_normal(n).astype(np.float32) * np.float32(sigma))
        dec = ref.step([g], 1.0)
        param.grad = torch.from_numpy((g.astype(np.uint32) << 16).view(np.float32).copy())
        total = float(torch.nn.utils.clip_grad_norm_([param], hp.max_grad_norm))
        topt.step()
        assert abs(dec.norm - total) <= 1e-6 * total
        clipped += dec.clip < 1.0
        unclipped += dec.clip == 1.0
    assert clipped >= 2 and unclipped >= 2
    # Two rounding orders differ by a few binary32 ulps of the intermediate
    # terms, which is hundreds of ulps of a result that cancels to near zero
    # (m changing sign, w crossing zero): bound the difference by the array's
    # RMS (measured at most 7e-6 of it) and the typical element's relative
    # error (measured 1e-7 to 8e-7). A dropped weight decay already moves w by
    # about 6e-5 of its RMS over these steps.
    st = topt.state[param]
    for mine, theirs in ((ref.w, param.detach()), (ref.m, st["exp_avg"]), (ref.v, st["exp_avg_sq"])):
        theirs = theirs.numpy().astype(np.float64)
        diff = np.abs(mine.astype(np.float64) - theirs)
        assert diff.max() <= 2e-5 * np.sqrt(np.mean(theirs * theirs)), diff.max()
        assert np.median(diff / np.maximum(np.abs(theirs), 1e-30)) <= 2e-6


def pin_params_are_bf16_of_new_weights(lib):
    """The all-gathered parameters are the updated master weights rounded to
    bf16 (Zero From Scratch, item 7: the all-gather hands every rank the
    updated parameters; the pages' mixed precision keeps them in bf16): after
    every applied step p equals PyTorch's round-to-nearest-even cast of the new
    w, bit for bit, and a skipped step leaves p as it was."""
    import torch

    rng = np.random.default_rng(23)
    n, p = 2048, 3
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    ref = _opt(lib, w0)
    for t in range(4):
        grads = [_trunc(rng.standard_normal(n).astype(np.float32) * np.float32(1e-3 * 1024)) for _ in range(p)]
        if t == 2:
            grads[1][5] = 0x7F80  # +inf: this step is skipped
        before = ref.p.copy()
        dec = ref.step(grads, 1024.0)
        if dec.found_inf:
            assert ref.p.tobytes() == before.tobytes()
        else:
            want = torch.from_numpy(ref.w.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert ref.p.tobytes() == want.tobytes()
            assert ref.p.tobytes() != before.tobytes()


def pin_clip_constant_vector(lib):
    """Every gradient element a: the norm is |a| sqrt(N)."""
    n, a = 4096, 0.125  # norm = 0.125 * 64 = 8
    g = _bf16(np.full(n, a, dtype=np.float32))
    opt = _opt(lib, np.zeros(n), weight_decay=0.0, max_grad_norm=1.0)
    d = opt.step([g], 1.0)
    assert d.norm == 8.0 and d.sumsq == 64.0
    want = 1.0 / (8.0 + 1e-6)
    assert abs(d.clip - want) <= _ulp(want)
    # clipped moment: m = (1 - beta1) * a * c
    assert np.allclose(opt.m, 0.1 * a * d.clip, rtol=2e-7)
    # below the threshold the factor is exactly one
    opt2 = _opt(lib, np.zeros(n), weight_decay=0.0, max_grad_norm=9.0)
    assert opt2.step([g], 1.0).clip == 1.0
    # the clipped gradient has norm max_norm * norm / (norm + 1e-6)
    assert abs(8.0 * d.clip - 8.0 / (8.0 + 1e-6)) <= 8.0 * _ulp(want)
    # the factor is the ratio taken in binary64 and rounded once to binary32:
    # for constant vectors the norm is exactly |a| * 64 (a^2 and the sum of
    # 4096 of them are exact), so the factor is known exactly for every a
    rng = np.random.default_rng(29)
    for a in _trunc(rng.uniform(0.02, 10.0, 24).astype(np.float32) * rng.choice([-1, 1], 24).astype(np.float32)):
        av = float((np.uint32(a) << np.uint32(16)).view(np.float32))
        d = _opt(lib, np.zeros(n), weight_decay=0.0, max_grad_norm=1.0).step([np.full(n, a, np.uint16)], 1.0)
        assert d.norm == abs(av) * 64.0
        assert d.clip == float(np.float32(1.0 / (abs(av) * 64.0 + 1e-6))), (av, d.clip)


def pin_norm_vs_fsum(lib):
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(200_003) * np.exp(rng.uniform(-8, 2, 200_003))).astype(np.float32)
    sq = (g * g).astype(np.float64)  # binary32 squares, widened
    exact = math.fsum(sq.tolist())
    got = oracle.sumsq(g, lib=lib)
    assert abs(got - exact) <= 1e-12 * exact, (got, exact)


def pin_average_and_unscale(lib):
    """Integer-valued gradients: every order of addition is exact, so the
    reduce-scatter + unscale must give exactly sum / (L * P)."""
    rng = np.random.default_rng(7)
    for p in (1, 2, 3, 4, 8, 16):
        n = 257
        ints = rng.integers(-64, 65, size=(p, n))
        L = 256.0
        grads = [_bf16((ints[r] * L).astype(np.float32)) for r in range(p)]
        inv = oracle.inv_scale(L, p, 1, lib=lib)
        g = oracle.reduce_unscale(grads, 0, n, inv, lib=lib)
        want = ints.sum(axis=0) / p  # exact in binary32 for these sizes only when P is 2^k
        if p & (p - 1) == 0:
            assert np.array_equal(g, want.astype(np.float32))
        else:
            assert np.allclose(g, want, rtol=2 * 2 ** -24, atol=0)
        inv_sum = oracle.inv_scale(L, p, 0, lib=lib)
        gs = oracle.reduce_unscale(grads, 0, n, inv_sum, lib=lib)
        assert np.array_equal(gs, ints.sum(axis=0).astype(np.float32))


def pin_skip_on_nonfinite(lib):
    rng = np.random.default_rng(9)
    n = 100
    for bad in (np.inf, -np.inf, np.nan):
        opt = _opt(lib, rng.standard_normal(n) * 0.02)
        good = _trunc(rng.standard_normal(n) * 1e-3)
        opt.step([good, good], 1024.0)
        snap = (opt.w.copy(), opt.m.copy(), opt.v.copy(), opt.p.copy(), opt.t)
        g2 = good.copy()
        g2[n - 1] = F32(bad).view(np.uint32) >> 16 if not np.isnan(bad) else 0x7FC0
        d = opt.step([good, g2], 1024.0)
        assert d.found_inf and opt.t == snap[4] and d.t == snap[4]
        for a, b in zip((opt.w, opt.m, opt.v, opt.p), snap[:4]):
            assert a.tobytes() == b.tobytes()
        d = opt.step([good, good], 1024.0)
        assert not d.found_inf and opt.t == snap[4] + 1


def pin_loss_scale_invariance(lib):
    """bf16(x * 2^k) = bf16(x) * 2^k, and the unscale undoes 2^k exactly."""
    rng = np.random.default_rng(21)
    n, p = 1000, 4
    x = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(p)]
    base = [_trunc(xi) for xi in x]
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    res = []
    for L in (1024.0, 65536.0):
        grads = [_bf16(oracle.bf16_to_f32(b) * F32(L)) for b in base]
        opt = _opt(lib, w0)
        for _ in range(3):
            opt.step(grads, L)
        res.append((opt.w.tobytes(), opt.m.tobytes(), opt.v.tobytes(), opt.p.tobytes()))
    assert res[0] == res[1]


# ------------------------------------------------------------- formats

def pin_bf16_rounding_vs_torch(lib):
    import torch

    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, size=40_000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, size=4000).astype(np.uint32) << 16) | 0x8000
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x7F7F8000, 0x00000001,
                        0x00008000, 0x00018000, 0x3F808000, 0x3F818000, 0xBF808000], dtype=np.uint32)
    bits = np.concatenate([u, ties, special])
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(x, lib=lib)
    assert np.array_equal(got, want)
    # NaN stays NaN (torch returns one canonical NaN, so only NaN-ness is
    # compared; the values reach the oracle as Python floats, already quiet)
    nan_bits = np.array([0x7F800001, 0x7F808000, 0x7FC00000, 0xFF800001, 0x7FFFFFFF, 0xFFBFFFFF], np.uint32)
    got_nan = oracle.f32_to_bf16(nan_bits.view(np.float32), lib=lib).astype(np.uint32) << np.uint32(16)
    assert np.all(np.isnan(got_nan.view(np.float32)))
    assert np.all(np.isnan(torch.from_numpy(nan_bits.view(np.float32).copy()).to(torch.bfloat16).float().numpy()))


def pin_e4m3_values_vs_torch(lib):
    import torch

    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([oracle.e4m3_value(int(c), lib=lib) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _e4m3_table():
    """Values of the non-negative finite codes 0x00..0x7E, from the format:
    exponent bias 7, 3 mantissa bits, subnormals at exponent field 0."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def nearest_e4m3(y: np.ndarray) -> np.ndarray:
    """Brute force: nearest table value, ties to the even code, sign kept."""
    tab = _e4m3_table()
    # Distances are exact in binary64 only for moderate magnitudes; every
    # magnitude above 448 has 448 as its nearest finite value, so cap there
    # (at 2^20, far above 448, which keeps the search itself deciding).
    a = np.minimum(np.abs(y), 2.0 ** 20)[:, None]
    dist = np.abs(a - tab[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among equal-distance candidates prefer the even code
    even = (np.arange(0x7F) % 2 == 0)[None, :]
    pick = np.where((cand & even).any(axis=1), np.argmax(cand & even, axis=1), np.argmax(cand, axis=1))
    return (pick | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def pin_e4m3_encoder_exhaustive(lib):
    """Every finite bf16 value as an encoder input, plus values around each
    rounding midpoint, against the brute-force nearest search."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    x32 = bits.view(np.float32)
    y = x32[np.isfinite(x32)].astype(np.float64)
    tab = _e4m3_table()
    mids = (tab[1:] + tab[:-1]) / 2
    around = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1), -mids, tab, -tab])
    ys = np.concatenate([y, around])
    got = np.array([oracle.e4m3_encode(v, lib=lib) for v in ys], dtype=np.uint8)
    for lo in range(0, ys.size, 8192):
        want = nearest_e4m3(ys[lo:lo + 8192])
        assert np.array_equal(got[lo:lo + 8192], want), lo


def pin_mx_scale_rule(lib):
    """Blocks built by hand from the OCP MX rule (e = floor(log2 amax) - 8)."""
    def block(vals):
        v = np.zeros(32, dtype=np.float32)
        v[: len(vals)] = vals
        return _bf16(v)

    for k in (-3, 0, 5):
        codes, sc = oracle.mx_encode(block([448.0 * 2.0 ** k, -1.0 * 2.0 ** k]), lib=lib)
        assert sc[0] == 127 + k and codes[0] == 0x7E and codes[1] == 0xB8  # -1.0 = 0x80|(7<<3)
        # the largest bf16 below 512 shares the binade and saturates to 448
        codes, sc = oracle.mx_encode(block([510.0 * 2.0 ** k]), lib=lib)
        assert sc[0] == 127 + k and codes[0] == 0x7E
        codes, sc = oracle.mx_encode(block([256.0 * 2.0 ** k]), lib=lib)
        assert sc[0] == 127 + k and codes[0] == 0x78
    # amax 1.0: e = -8; 2^-17 -> y = 2^-9 (smallest subnormal); 2^-18 -> tie -> 0;
    # 3 * 2^-19 -> y = 1.5 * 2^-10 -> 2^-9; -2^-20 -> -0
    codes, sc = oracle.mx_encode(block([1.0, 2.0 ** -17, 2.0 ** -18, 3 * 2.0 ** -19, -(2.0 ** -20)]), lib=lib)
    assert sc[0] == 119
    assert list(codes[:5]) == [0x78, 0x01, 0x00, 0x01, 0x80]  # 1.0 * 2^8 = 256 -> 0x78
    # all zero, and negative zero keeps its sign
    z = block([])
    z[3] = 0x8000
    codes, sc = oracle.mx_encode(z, lib=lib)
    assert sc[0] == 0 and codes[3] == 0x80 and codes[0] == 0
    # bf16 subnormals only: the scale clamps at 2^-127, 2^-133 * 2^127 = 2^-6
    sub = np.zeros(32, dtype=np.uint16)
    sub[0], sub[1] = 0x0001, 0x0040  # 2^-133 and 2^-127
    codes, sc = oracle.mx_encode(sub, lib=lib)
    assert sc[0] == 0 and codes[0] == 0x08 and codes[1] == 0x38  # 2^-6 and 2^0
    # any infinity or NaN poisons the block
    for bad in (0x7F80, 0xFF80, 0x7FC0):
        x = block([1.0])
        x[7] = bad
        codes, sc = oracle.mx_encode(x, lib=lib)
        assert sc[0] == 0xFF and np.all(codes == 0x7F)
        assert math.isnan(oracle.mx_decode(0x00, 0xFF, lib=lib))
    # a ragged tail block: missing elements count as zero; amax 3 -> e = -7,
    # 3 * 2^7 = 384 = 1.5 * 2^8 -> 0x7C, -0.5 * 2^7 = -2^6 -> 0x80 | (13 << 3)
    codes, sc = oracle.mx_encode(_bf16(np.array([3.0, -0.5], dtype=np.float32)), lib=lib)
    assert sc.size == 1 and sc[0] == 127 - 7 and list(codes) == [0x7C, 0xE8]
    # decode multiplies by 2^(s-127), down to the subnormal scale 2^-127
    assert oracle.mx_decode(0x01, 0, lib=lib) == 2.0 ** -136
    assert oracle.mx_decode(0x7E, 246, lib=lib) == 448.0 * 2.0 ** 119


def pin_mx_roundtrip_error_bound(lib):
    """Decoding an encoded block returns every value to within half an E4M3
    spacing at the block's scale (spacing 2^(floor(log2 |y|) - 3) for normal
    magnitudes, 2^-9 below 2^-6, where y = x 2^-e), or saturates exactly to
    448 2^e; the scale follows the block's largest magnitude (e = floor(log2
    amax) - 8). Random blocks over sixty binades, signs mixed, zeros
    included: a bound from the format definition, not a second encoder."""
    rng = np.random.default_rng(37)
    nblk = 400
    mag = np.exp2(rng.uniform(-30, 30, nblk))[:, None] * np.exp2(rng.uniform(-12, 0, (nblk, 32)))
    x = (mag * rng.choice([-1.0, 1.0], (nblk, 32))).astype(np.float32)
    x[rng.random((nblk, 32)) < 0.05] = 0.0
    xb = _trunc(x.ravel())
    xv = (xb.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64).reshape(nblk, 32)
    codes, scales = oracle.mx_encode(xb, lib=lib)
    for b in range(nblk):
        amax = np.max(np.abs(xv[b]))
        e = int(scales[b]) - 127
        if amax == 0.0:
            assert scales[b] == 0
            continue
        assert e == max(-127, min(127, math.floor(math.log2(amax)) - 8)), (b, e, amax)
        for j in range(32):
            y = xv[b, j] * 2.0 ** -e
            d = oracle.mx_decode(int(codes[32 * b + j]), int(scales[b]), lib=lib) * 2.0 ** -e
            assert not math.isnan(d)
            if abs(y) > 448.0:
                assert d == math.copysign(448.0, y), (b, j, y, d)
            else:
                spacing = 2.0 ** (math.floor(math.log2(abs(y))) - 3) if abs(y) >= 2.0 ** -6 else 2.0 ** -9
                assert abs(d - y) <= spacing / 2, (b, j, y, d)


def pin_mx_loss_scale_shifts_scale_only(lib):
    import zero_sharded_mixed_flat_gb300.synth as synth

    x = synth.random_bf16(32 * 50, seed=4, scale=1e-3, dist="student_t")
    xf = oracle.bf16_to_f32(x)
    c1, s1 = oracle.mx_encode(x, lib=lib)
    c2, s2 = oracle.mx_encode(_bf16(xf * F32(1024.0)), lib=lib)
    assert np.array_equal(c1, c2)
    assert np.array_equal(s2.astype(int) - s1.astype(int), np.full(s1.size, 10))


def pin_mx_f32_encoder(lib):
    """The MX block rule on fp32 values (stored MX parameters)."""
    f32 = lambda v: np.array(v, dtype=np.float32)
    # amax 1.0 -> e = -8, y = 256 x. 1 + 2^-4 -> y = 272, a tie between 256 and
    # 288 -> even -> 256 (0x78); one fp32 ulp more breaks the tie upwards.
    x = np.zeros(32, np.float32)
    x[:3] = [1.0, 1.0 + 2.0 ** -4, np.nextafter(F32(1.0 + 2.0 ** -4), F32(2.0))]
    codes, sc = oracle.mx_encode_f32(x, lib=lib)
    assert sc[0] == 119 and list(codes[:3]) == [0x78, 0x78, 0x79]
    # largest finite fp32 binade: e = 127 - 8 = 119, byte 246
    codes, sc = oracle.mx_encode_f32(f32([3.0e38, -1.0e38]), lib=lib)
    assert sc[0] == 246 and codes[0] == 0x7E and codes[1] & 0x80
    # an fp32-subnormal block clamps at 2^-127: 2^-140 * 2^127 = 2^-13 -> 0;
    # -2^-135 * 2^127 = -2^-8 = -(2 * 2^-9), the subnormal code 0x82; the
    # smallest fp32 subnormal -2^-149 -> -2^-22 -> -0
    codes, sc = oracle.mx_encode_f32(f32([2.0 ** -140, -(2.0 ** -135), -(2.0 ** -149)]), lib=lib)
    assert sc[0] == 0 and list(codes[:3]) == [0x00, 0x82, 0x80]
    # non-finite poisons the block
    codes, sc = oracle.mx_encode_f32(f32([1.0, np.inf, 2.0]), lib=lib)
    assert sc[0] == 0xFF and np.all(codes == 0x7F)
    # on bf16-representable values it agrees with the bf16 encoder
    xb = (np.random.default_rng(2).standard_normal(32 * 40).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    a = oracle.mx_encode(xb, lib=lib)
    b = oracle.mx_encode_f32(oracle.bf16_to_f32(xb), lib=lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # random fp32 blocks over many binades: each code is the nearest E4M3 value
    # (ties to even) of x * 2^-e, with e from the block's amax
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(32 * 300) * np.exp(rng.uniform(-30, 30, 32 * 300))).astype(np.float32)
    x = x[:32 * 299 + 7]  # a ragged last block
    codes, sc = oracle.mx_encode_f32(x, lib=lib)
    for blk in range(sc.size):
        v = x[32 * blk:32 * blk + 32].astype(np.float64)
        k = np.frexp(np.max(np.abs(v)))[1]
        e = int(np.clip(k - 1 - 8, -127, 127))
        assert sc[blk] == e + 127
        assert np.array_equal(codes[32 * blk:32 * blk + v.size], nearest_e4m3(np.ldexp(v, -e)))


# ------------------------------------------------------------- sharding

def pin_shard_layout(lib):
    for n in (1, 31, 32, 33, 1000, 65_549, 124_439_808, 3_000_000_000):
        for p in (1, 2, 3, 4, 7, 8, 16):
            s = oracle.shard_len(n, p, lib=lib)
            assert s % 32 == 0 and p * s >= n and s >= -(-n // p) and s < -(-n // p) + 32


def pin_identical_learning(lib):
    """Zero From Scratch, item 19: the sharded (stage-two) step learns exactly
    what the unsharded step learns, for every P, over ten steps."""
    rng = np.random.default_rng(13)
    n = 1013
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    for p in (1, 2, 3, 4, 8):
        a = _opt(lib, w0, max_grad_norm=0.0)
        b = _opt(lib, w0, max_grad_norm=0.0)
        for _ in range(10):
            grads = [_trunc(rng.standard_normal(n) * 1e-3 * 1024) for _ in range(p)]
            da = a.step(grads, 1024.0)
            db = b.step(grads, 1024.0, sharded=True)
            assert da.found_inf == db.found_inf
            assert abs(da.sumsq - db.sumsq) <= 1e-13 * da.sumsq
        for x, y in ((a.w, b.w), (a.m, b.m), (a.v, b.v), (a.p, b.p)):
            assert x.tobytes() == y.tobytes(), p
        assert a.t == b.t == 10


def pin_resume(lib):
    rng = np.random.default_rng(17)
    n, p = 300, 2
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    steps = [[_trunc(rng.standard_normal(n)) for _ in range(p)] for _ in range(10)]
    full = _opt(lib, w0)
    for g in steps:
        full.step(g, 1024.0)
    first = _opt(lib, w0)
    for g in steps[:6]:
        first.step(g, 1024.0)
    resumed = _opt(lib, first.w)
    resumed.m[:], resumed.v[:] = first.m, first.v
    resumed.set_step(first.t)
    for g in steps[6:]:
        resumed.step(g, 1024.0)
    for x, y in ((full.w, resumed.w), (full.m, resumed.m), (full.v, resumed.v), (full.p, resumed.p)):
        assert x.tobytes() == y.tobytes()
    t, b1p, b2p = oracle.counters_at(oracle.Hparams(), 10, lib=lib)
    assert t == 10 and abs(b1p - 0.9 ** 10) <= 1e-15 and abs(b2p - 0.999 ** 10) <= 1e-15


def _ranges(s: int, p: int):
    """Gather ranges that start and end on, next to and away from shard edges."""
    n = p * s
    edges = sorted({0, 1, s - 1, s, s + 1, n // 2, n - s - 1, n - s, n - 1, n} & set(range(n + 1)))
    return [(lo, hi) for lo in edges for hi in edges if hi >= lo]


def pin_gather_owner_offset(lib):
    """Stage three's gather (DeepSpeed documentation review, paragraph on the
    stages): with every rank's shard holding its own flat indices as values,
    a gathered range must read back as the indices themselves."""
    for p, s in ((1, 32), (2, 32), (3, 64), (5, 32), (8, 96)):
        shards = [np.arange(r * s, (r + 1) * s, dtype=np.uint16) for r in range(p)]
        for lo, hi in _ranges(s, p):
            got = oracle.gather(shards, s, lo, hi, lib=lib)
            assert np.array_equal(got, np.arange(lo, hi, dtype=np.uint16)), (p, s, lo, hi)


def pin_gather_mx_hand_values(lib):
    """MX parameter shards built by hand from the formats: E4M3 (bias 7,
    subnormals m/8 * 2^-6), E8M0 scale 2^(s - 127), bf16 with round to nearest
    even, whose subnormal step is 2^-133."""
    s = 96
    codes = [np.zeros(s, np.uint8), np.zeros(s, np.uint8)]
    scales = [np.array([119, 0, 127], np.uint8), np.array([120, 127, 0xFF], np.uint8)]
    want = np.zeros(2 * s, np.uint16)
    want[2 * s - 32:] = 0x7FC0  # a NaN scale: the whole block gathers as NaN
    cases = [  # (rank, index in shard, code, expected bf16)
        (0, 0, 0x78, 0x3F80),   # 256 * 2^-8 = 1
        (0, 1, 0xF8, 0xBF80),   # -1
        (0, 2, 0x80, 0x8000),   # -0 keeps its sign
        (0, 3, 0x7F, 0x7FC0),   # NaN code
        (0, 32, 0x05, 0x0001),  # 5 * 2^-136 = 0.625 subnormal steps -> 1
        (0, 33, 0x04, 0x0000),  # 0.5 steps: tie to even -> 0
        (0, 34, 0x0C, 0x0002),  # 1.5 * 2^-6 * 2^-127 = 1.5 steps: tie to even -> 2
        (0, 35, 0x84, 0x8000),  # -0.5 steps -> -0
        (1, 0, 0x78, 0x4000),   # 256 * 2^-7 = 2: rank one's own scale
        (1, 32, 0x7E, 0x43E0),  # 448
        (1, 33, 0x01, 0x3B00),  # 2^-9
        (1, 34, 0xB9, 0xBF90),  # exponent field 7: -(1 + 1/8) * 2^0 = -1.125
    ]
    for r, k, c, b in cases:
        codes[r][k] = c
        want[r * s + k] = b
    for lo, hi in _ranges(s, 2) + [(30, 40), (s - 3, s + 40)]:
        got = oracle.gather_mx(codes, scales, s, lo, hi, lib=lib)
        assert np.array_equal(got, want[lo:hi]), (lo, hi, got, want[lo:hi])


def pin_gather_mx_vs_torch(lib):
    """Random MX shards decoded through torch's float8_e4m3fn values, an
    exact power-of-two scaling and torch's bf16 cast."""
    import torch

    rng = np.random.default_rng(23)
    p, s = 3, 4096
    codes, scales = [], []
    for _ in range(p):
        c = rng.integers(0, 256, s).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x3C  # no NaN codes here
        codes.append(c)
        scales.append(np.concatenate([rng.integers(100, 150, s // 32 - 8), rng.integers(0, 8, 8)]).astype(np.uint8))
    flat_vals = []
    for c, sc in zip(codes, scales):
        v = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
        flat_vals.append(np.ldexp(v, np.repeat(sc.astype(np.int64) - 127, 32)).astype(np.float32))
    ref = torch.from_numpy(np.concatenate(flat_vals)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for lo, hi in ((0, p * s), (5, 4100), (4096, 8192), (8000, 12288)):
        assert np.array_equal(oracle.gather_mx(codes, scales, s, lo, hi, lib=lib), ref[lo:hi]), (lo, hi)


def pin_mx_reduce_vs_torch_decode(lib):
    """The MX reduce-scatter: each rank's codes decoded through torch's
    float8_e4m3fn values and an exact power-of-two scaling, added in rank
    order in binary32 (numpy), then unscaled; bit for bit."""
    import torch

    rng = np.random.default_rng(29)
    n, p = 4096, 5
    codes, scales, vals = [], [], []
    for _ in range(p):
        c = rng.integers(0, 256, n).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x21  # finite codes only
        sc = rng.integers(100, 150, n // 32).astype(np.uint8)
        sc[rng.choice(n // 32, 6, replace=False)] = 0  # subnormal scale
        codes.append(c)
        scales.append(sc)
        v = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
        vals.append(np.ldexp(v, np.repeat(sc.astype(np.int64) - 127, 32)).astype(np.float32))
    acc = np.zeros(n, np.float32)
    for v in vals:
        acc = (acc + v).astype(np.float32)
    inv = np.float32(1.0 / (1024.0 * p))
    want = (acc * inv).astype(np.float32)
    got = oracle.mx_reduce_unscale(codes, scales, 0, n, float(inv), lib=lib)
    assert got.tobytes() == want.tobytes()
    got = oracle.mx_reduce_unscale(codes, scales, 100, 3000, float(inv), lib=lib)
    assert got.tobytes() == want[100:3000].tobytes()


def pin_mx_step_lossless_equals_bf16_step(lib):
    """Gradients whose every value is exactly an E4M3 value times its block's
    scale (each block's values are +-(1 + k/8) 2^j, k <= 6, within six binades
    of the block maximum, which has the block's top exponent) encode without loss,
    so the MX step must equal the bf16 step on the same values bit for bit."""
    rng = np.random.default_rng(31)
    n, p, L = 4096, 3, 1024.0

    def lossless(seed):
        r = np.random.default_rng(seed)
        x = np.empty(n, np.float32)
        for b in range(n // 32):
            top = int(r.integers(-5, 3))
            k = r.integers(0, 7, 32)  # E4M3's top binade ends at 1.75 (mantissa 111 there is NaN)
            d = r.integers(0, 7, 32)
            d[0] = 0  # one value carries the block's top exponent
            x[32 * b:32 * b + 32] = (r.choice([-1.0, 1.0], 32) * (1 + k / 8) * 2.0 ** (top - d)).astype(np.float32)
        return _bf16(x)

    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    a, b = _opt(lib, w0), _opt(lib, w0)
    for t in range(3):
        grads = [lossless(100 * t + r) for r in range(p)]
        enc = [oracle.mx_encode(g, lib=lib) for g in grads]
        for g, (c, sc) in zip(grads, enc):  # the encoding is lossless
            dec = np.array([oracle.mx_decode(c[i], sc[i // 32], lib=lib) for i in range(0, n, 97)], np.float32)
            assert np.array_equal(dec, (g[::97].astype(np.uint32) << 16).view(np.float32))
        da = a.step(grads, L)
        db = b.step_mx([c for c, _ in enc], [sc for _, sc in enc], L)
        assert da.sumsq == db.sumsq and da.clip == db.clip
    for x, y in ((a.w, b.w), (a.m, b.m), (a.v, b.v), (a.p, b.p)):
        assert x.tobytes() == y.tobytes()


PINS = [
    pin_first_step_closed_form,
    pin_first_step_weight_decay,
    pin_constant_gradient,
    pin_two_step_closed_form,
    pin_adamw_and_clip_vs_torch,
    pin_params_are_bf16_of_new_weights,
    pin_clip_constant_vector,
    pin_norm_vs_fsum,
    pin_average_and_unscale,
    pin_skip_on_nonfinite,
    pin_loss_scale_invariance,
    pin_bf16_rounding_vs_torch,
    pin_e4m3_values_vs_torch,
    pin_e4m3_encoder_exhaustive,
    pin_mx_scale_rule,
    pin_mx_loss_scale_shifts_scale_only,
    pin_mx_roundtrip_error_bound,
    pin_mx_f32_encoder,
    pin_shard_layout,
    pin_identical_learning,
    pin_resume,
    pin_gather_owner_offset,
    pin_gather_mx_hand_values,
    pin_gather_mx_vs_torch,
    pin_mx_reduce_vs_torch_decode,
    pin_mx_step_lossless_equals_bf16_step,
]


def run_all(lib) -> list[str]:
    """Run every pin; return the names of those that failed (used on mutants)."""
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except Exception:  # a mutant may also raise instead of failing an assert
            failed.append(pin.__name__)
    return failed
