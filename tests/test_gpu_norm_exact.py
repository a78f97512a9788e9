"""The norm pass's sum of squares: exact over its chunk sums, rounded once.

The norm pass hands out chunks of 32 eight-element vectors to warps as they
come free, and adds each chunk's sum of squares (a pair of binary32 values)
exactly into a fixed-point accumulator before rounding the total once to
binary64, so the result cannot depend on which warp took which chunk. These
tests pin that arithmetic from outside the library:

- where every chunk's sum is itself exact in binary32 (squares of small
  integers times a power of two that changes from chunk to chunk, spread
  over some 260 binades, from binary32 denormal squares up to chunks whose
  binary32 sum overflows and are added square by square), the sum of
  squares equals the correctly rounded sum of all squares (math.fsum), bit
  for bit, where a running binary64 sum would lose the small chunks;
- on ordinary gradients it is within 2^-40 of the correctly rounded sum of
  the binary32 squares, and within 1e-12 of the oracle's running binary64 sum;
- a NaN square anywhere gives NaN, an infinite square (and no NaN) +inf, as
  IEEE addition would, and the step is refused either way;
- repeating a norm pass gives the same bits.
"""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import to_dev_bf16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

CHUNK = 256  # elements per warp chunk (32 vectors of 8)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 values that bf16 holds exactly, as bf16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _sumsq(ctx, grads, loss_scale: float) -> float:
    zb.zg_grad_norm(ctx, grads, loss_scale)
    return zb.zg_get_info(ctx).sumsq


@pytest.mark.parametrize("p", [1, 2])
def test_sum_is_exact_over_wide_magnitudes(p):
    """Chunk c holds k * 2^e_c with |k| <= 15 and e_c from -74 to 59: every
    binary32 square k^2 * 2^(2 e_c) is exact (denormal below 2^-126), and so
    is each chunk's binary32 sum, except the chunks whose sum overflows
    binary32 (e_c = 59), which the pass adds square by square. With P = 2
    both ranks hold the same values: the rank sum 2g times 1/2 is exact."""
    rng = np.random.default_rng(12 + p)
    nchunk = 700
    n = nchunk * CHUNK + 5
    e = rng.integers(-74, 57, nchunk)
    e[[3, 400]] = 59  # binary32 chunk sums overflow here
    e[[10, 11, 650]] = -74  # denormal squares
    ex = np.concatenate([np.repeat(e, CHUNK), np.zeros(5, dtype=np.int64)])
    k = rng.integers(-15, 16, n)
    k[3 * CHUNK:4 * CHUNK] = 15
    g = (k * np.exp2(ex.astype(np.float64))).astype(np.float32)
    assert np.all(np.isfinite(g * g))
    bits = _bf16_bits(g)
    want = math.fsum((g.astype(np.float64) ** 2).tolist())
    ctx = zb.zg_init(n, p)
    grads = [to_dev_bf16(bits) for _ in range(p)]
    got = _sumsq(ctx, grads, 1.0)
    assert got == want, (got, want, got - want)


@pytest.mark.parametrize("n,p", [(1, 1), (7, 3), (4099, 4), ((1 << 20) + 13, 8), (3_000_017, 16)])
def test_sum_tracks_the_correctly_rounded_sum(n, p):
    host = [synth.random_bf16(n, seed=900 + 7 * r + n % 97, scale=1e-3 * 1024.0) for r in range(p)]
    g = oracle.reduce_unscale(host, 0, n, oracle.inv_scale(1024.0, p))
    sq = (g * g).astype(np.float64)  # binary32 squares, exact in binary64
    want = math.fsum(sq.tolist())
    ctx = zb.zg_init(n, p)
    grads = [to_dev_bf16(h) for h in host]
    got = _sumsq(ctx, grads, 1024.0)
    assert abs(got - want) <= 2.0 ** -40 * want, (n, p, got, want)
    ref = oracle.sumsq(g)
    assert abs(got - ref) <= 1e-12 * ref, (n, p, got, ref)
    assert _sumsq(ctx, grads, 1024.0) == got  # same gradients, same bits


@pytest.mark.parametrize("plant", ["inf", "nan", "both", "square_overflow"])
def test_non_finite_squares(plant):
    n, p = 70_001, 2
    host = [synth.random_bf16(n, seed=40 + r, scale=1.0) for r in range(p)]
    if plant in ("inf", "both"):
        host[0][12_345] = 0x7F80
    if plant in ("nan", "both"):
        host[1][n - 1] = 0x7FC0
    if plant == "square_overflow":
        host[0][500] = host[1][500] = 0x5F80  # 2^64: finite, its binary32 square is not
    ctx = zb.zg_init(n, p)
    got = _sumsq(ctx, [to_dev_bf16(h) for h in host], 1.0)
    info = zb.zg_get_info(ctx)
    assert info.found_inf == 1
    if plant in ("nan", "both"):
        assert math.isnan(got), got
    else:
        assert got == math.inf, got
    # the next, finite call is right again (the pass left its work array clear)
    clean = [synth.random_bf16(n, seed=60 + r, scale=1.0) for r in range(p)]
    got = _sumsq(ctx, [to_dev_bf16(h) for h in clean], 1.0)
    want = math.fsum((oracle.reduce_unscale(clean, 0, n, oracle.inv_scale(1.0, p)) ** 2).astype(np.float64).tolist())
    assert abs(got - want) <= 2.0 ** -40 * want and zb.zg_get_info(ctx).found_inf == 0
