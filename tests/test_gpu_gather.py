"""Stage three's just-in-time parameter gather on the GPU vs the oracle
(DeepSpeed documentation review, paragraph on the three stages: parameters
split across ranks, gathered for each layer's computation).

The P shards are separate guarded device buffers, or the parameter vector
itself cut at multiples of S. Every gathered range must equal the oracle's
gather bit for bit: across shard edges, ragged tails, starts off the vector
alignment, empty ranges and the whole vector. Canaries around the output
catch writes past it, and the padding past N in the last shards holds NaN
patterns that would show if a gather read them."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Guarded, log, to_dev_bf16, to_host_u16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

POISON_BF16 = 0x7FC1
SIZES = [(1, 1), (31, 2), (1000, 3), (4099, 4), (65_549, 4), (30_001, 5), (77_777, 11), (65_536, 16), (200_003, 8),
         ((1 << 20) + 40, 8)]


def ranges(n: int, s: int, seed: int, extra: int = 40):
    """Edges of shards, of 8- and 16-element vectors and of the vector, in
    every combination, plus random ranges."""
    marks = {0, 1, 7, 8, 9, 15, 16, 17, 31, 33, s - 1, s, s + 1, s + 8, s + 16, 2 * s - 1, 2 * s + 3, n // 2,
             n - 17, n - 16, n - 9, n - 8, n - 1, n}
    marks = sorted(m for m in marks if 0 <= m <= n)
    out = [(a, b) for a in marks for b in marks if b >= a]
    rng = np.random.default_rng(seed)
    for _ in range(extra):
        a, b = sorted(rng.integers(0, n + 1, 2).tolist())
        out.append((a, b))
    return out


def bf16_shards(n: int, p: int, seed: int):
    s = oracle.shard_len(n, p)
    host = []
    for r in range(p):
        h = synth.random_bf16(s, seed=seed + r, scale=0.02)
        h[max(0, min(s, n - r * s)):] = POISON_BF16  # padding past N: never read
        host.append(h)
    dev = []
    for h in host:
        g = Guarded(s, torch.bfloat16)
        to_dev_bf16(h, g.view)
        dev.append(g)
    return s, host, dev


@pytest.mark.parametrize("how", ["kernel", "dma"])
@pytest.mark.parametrize("n,p", SIZES)
def test_gather_bf16_matches_oracle(n, p, how):
    fn = zb.zg_gather_params if how == "kernel" else zb.zg_gather_params_dma
    ctx = zb.zg_init(n, p)
    s, host, dev = bf16_shards(n, p, seed=n + 7 * p)
    assert s == zb.zg_shard_len(ctx)
    out = Guarded(n, torch.bfloat16)
    checked = 0
    for lo, hi in ranges(n, s, seed=n):
        out.view.fill_(-1.0)
        fn(ctx, [d.view for d in dev], lo, hi, out.view[:hi - lo])
        got = to_host_u16(out.view)
        want = oracle.gather(host, s, lo, hi)
        assert np.array_equal(got[:hi - lo], want), (n, p, lo, hi, np.nonzero(got[:hi - lo] != want)[0][:5])
        assert np.all(got[hi - lo:] == 0xBF80), (n, p, lo, hi)  # -1.0 left alone past the range
        assert out.intact() and all(d.intact() for d in dev), (n, p, lo, hi)
        checked += 1
    log({"case": f"gather bf16 ({how}) n={n} p={p}", "ranges": checked, "bitexact": 1.0})


@pytest.mark.parametrize("n,p", SIZES)
def test_gather_mx_matches_oracle(n, p):
    """Random code and scale bytes (every pattern, NaN codes and the NaN and
    subnormal scales included): the gather is a decode of whatever it holds."""
    ctx = zb.zg_init(n, p)
    s = zb.zg_shard_len(ctx)
    rng = np.random.default_rng(n * 31 + p)
    codes = [rng.integers(0, 256, s).astype(np.uint8) for _ in range(p)]
    scales = [rng.integers(0, 256, s // 32).astype(np.uint8) for _ in range(p)]
    for sc in scales:
        sc[: min(4, sc.size)] = [0, 1, 254, 255][: min(4, sc.size)]
    dc = [Guarded(s, torch.uint8) for _ in range(p)]
    ds = [Guarded(s // 32, torch.uint8) for _ in range(p)]
    for g, h in zip(dc + ds, codes + scales):
        g.view.copy_(torch.from_numpy(h))
    out = Guarded(n, torch.bfloat16)
    checked = 0
    for lo, hi in ranges(n, s, seed=n + 1):
        out.view.fill_(-1.0)
        zb.zg_gather_params_mxfp8(ctx, [g.view for g in dc], [g.view for g in ds], lo, hi, out.view[:hi - lo])
        got = to_host_u16(out.view)
        want = oracle.gather_mx(codes, scales, s, lo, hi)
        assert np.array_equal(got[:hi - lo], want), (n, p, lo, hi, np.nonzero(got[:hi - lo] != want)[0][:5])
        assert np.all(got[hi - lo:] == 0xBF80), (n, p, lo, hi)
        assert out.intact() and all(g.intact() for g in dc + ds), (n, p, lo, hi)
        checked += 1
    log({"case": f"gather mx n={n} p={p}", "ranges": checked, "bitexact": 1.0})


@pytest.mark.parametrize("mx", [False, True])
def test_gather_after_steps(mx):
    """The optimizer's own parameter vector, cut into its P shards: the whole
    gather returns the vector (all-gather of the shards = the replicated
    parameters), and any layer range equals the oracle's gather of what the
    step wrote."""
    n, p = 200_003, 8
    w0 = torch.from_numpy((np.random.default_rng(3).standard_normal(n) * 0.02).astype(np.float32))
    opt = zb.ShardedAdamW(n, p, zb.Hparams(), w0)
    if mx:
        opt.use_mx_params()
    for k in range(2):
        grads = [to_dev_bf16(synth.random_bf16(n, seed=50 + 10 * k + r, scale=1e-3 * 1024)) for r in range(p)]
        opt.step(grads, 1024.0)
    assert opt.info().step_t == 2
    s = opt.shard_len
    full = to_host_u16(opt.gather(0, n))
    if mx:
        c = opt.pcodes.cpu().numpy()
        sc = opt.pscales.cpu().numpy()
        cs = [np.pad(c[r * s:(r + 1) * s], (0, s - c[r * s:(r + 1) * s].size)) for r in range(p)]
        ss = [np.pad(sc[r * s // 32:(r + 1) * s // 32], (0, s // 32 - sc[r * s // 32:(r + 1) * s // 32].size))
              for r in range(p)]
        assert np.array_equal(full, oracle.gather_mx(cs, ss, s, 0, n))
        # decoded MX parameters sit within the E4M3 step of the master weights
        w = opt.w.cpu().numpy()
        dec = torch.from_numpy(full.view(np.int16)).view(torch.bfloat16).float().numpy()
        amax = np.abs(np.pad(w, (0, -n % 32))).reshape(-1, 32).max(axis=1).repeat(32)[:n]
        assert np.all(np.abs(dec - w) <= amax * 2.0 ** -3)
    else:
        params = to_host_u16(opt.params)
        assert np.array_equal(full, params)
        shards = [np.pad(params[r * s:(r + 1) * s], (0, s - params[r * s:(r + 1) * s].size)) for r in range(p)]
        for lo, hi in ((0, 768), (768, 768 * 5), (s - 100, s + 100), (n - 1000, n), (12_345, 150_001)):
            assert np.array_equal(to_host_u16(opt.gather(lo, hi)), oracle.gather(shards, s, lo, hi)), (lo, hi)


def test_gather_gpt2_layers_full_size():
    """N = 124,439,808 at P = 8 (the GPT-2-small parameter vector): every one
    of the 148 tensors gathered at its offset rebuilds the vector bit for bit;
    MX shards of the same size decode like the oracle on sampled tensors."""
    wl = synth.workload("gpt2small_p8")
    n, p = wl.n, wl.p
    ctx = zb.zg_init(n, p)
    s = zb.zg_shard_len(ctx)
    gen = torch.Generator(device="cuda").manual_seed(11)
    params = torch.randint(-32768, 32768, (p * s,), dtype=torch.int32, device="cuda", generator=gen)
    params = params.to(torch.int16).view(torch.bfloat16)
    out = torch.full((n,), -1.0, dtype=torch.bfloat16, device="cuda")
    sizes = [k for _, k in synth.gpt2_small_tensors()]
    offsets = np.concatenate([[0], np.cumsum(sizes)])
    for lo, hi in zip(offsets[:-1], offsets[1:]):
        zb.zg_gather_params(ctx, params, int(lo), int(hi), out[lo:hi])
    assert torch.equal(out.view(torch.int16), params[:n].view(torch.int16))
    # MX: random bytes, sampled tensors against the oracle
    codes = torch.randint(0, 256, (p * s,), dtype=torch.int32, device="cuda", generator=gen).to(torch.uint8)
    scales = torch.randint(100, 160, (p * s // 32,), dtype=torch.int32, device="cuda", generator=gen).to(torch.uint8)
    hc = codes.cpu().numpy()
    hs = scales.cpu().numpy()
    cs = [hc[r * s:(r + 1) * s] for r in range(p)]
    ss = [hs[r * s // 32:(r + 1) * s // 32] for r in range(p)]
    picks = [0, 1, 2, 50, 77, 146, 147]  # wte, wpe, ln_1, mid-stack, ln_f
    for t in picks:
        lo, hi = int(offsets[t]), int(offsets[t + 1])
        o = torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda")
        zb.zg_gather_params_mxfp8(ctx, codes, scales, lo, hi, o)
        assert np.array_equal(to_host_u16(o), oracle.gather_mx(cs, ss, s, lo, hi)), t
    # a range that straddles shard edges and starts off the vector alignment
    lo, hi = s - 1_000_003, 3 * s + 77
    o = torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda")
    zb.zg_gather_params_mxfp8(ctx, codes, scales, lo, hi, o)
    assert np.array_equal(to_host_u16(o), oracle.gather_mx(cs, ss, s, lo, hi))
    zb.zg_gather_params(ctx, params, lo, hi, o)
    assert np.array_equal(to_host_u16(o), to_host_u16(params[lo:hi]))


def test_gather_argument_errors():
    n, p = 4096, 4
    ctx = zb.zg_init(n, p)
    s = zb.zg_shard_len(ctx)
    params = torch.zeros(p * s, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    L = zb.lib()
    ptrs = zb._ptr_array([params.data_ptr() + 2 * r * s for r in range(p)])
    assert L.zg_gather_params(ctx.handle, ptrs, 0, n + 1, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params(ctx.handle, ptrs, 10, 9, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params(ctx.handle, ptrs, -1, 9, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params(ctx.handle, ptrs, 0, 16, None, None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params(ctx.handle, ptrs, 0, 16, out.data_ptr() + 2, None) == zb.ZG_ERR_MISALIGNED
    assert L.zg_gather_params(ctx.handle, ptrs, 5, 5, None, None) == zb.ZG_OK  # empty: nothing to do
    bad = zb._ptr_array([params.data_ptr() + 2 * r * s + (2 if r == 2 else 0) for r in range(p)])
    assert L.zg_gather_params(ctx.handle, bad, 0, 16, out.data_ptr(), None) == zb.ZG_ERR_MISALIGNED
    null = zb._ptr_array([params.data_ptr() if r != 1 else 0 for r in range(p)])
    assert L.zg_gather_params(ctx.handle, null, 0, 16, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params(ctx.handle, None, 0, 16, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params_dma(ctx.handle, ptrs, 0, n + 1, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params_dma(ctx.handle, ptrs, 0, 16, out.data_ptr() + 2, None) == zb.ZG_ERR_MISALIGNED
    assert L.zg_gather_params_dma(ctx.handle, null, 0, 16, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params_dma(ctx.handle, ptrs, 7, 7, None, None) == zb.ZG_OK
    codes = torch.zeros(p * s, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(p * s // 32, dtype=torch.uint8, device="cuda")
    cp = zb._ptr_array([codes.data_ptr() + r * s for r in range(p)])
    sp = zb._ptr_array([scales.data_ptr() + r * s // 32 for r in range(p)])
    assert L.zg_gather_params_mxfp8(ctx.handle, cp, sp, 0, n + 1, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    assert L.zg_gather_params_mxfp8(ctx.handle, cp, None, 0, 16, out.data_ptr(), None) == zb.ZG_ERR_INVALID_ARG
    cbad = zb._ptr_array([codes.data_ptr() + r * s + (1 if r == 3 else 0) for r in range(p)])
    assert L.zg_gather_params_mxfp8(ctx.handle, cbad, sp, 0, 16, out.data_ptr(), None) == zb.ZG_ERR_MISALIGNED
    # scales need no alignment
    sodd = zb._ptr_array([scales.data_ptr() + 1 + r * (s // 32 - 1) for r in range(p)])
    assert L.zg_gather_params_mxfp8(ctx.handle, cp, sodd, 0, 16, out.data_ptr(), None) == zb.ZG_OK
    torch.cuda.synchronize()


def test_gather_in_cuda_graph():
    """A gather allocates nothing and makes no host round trip, so a layer
    loop of gathers captures into a CUDA graph; each replay reads the shards
    as they are then."""
    n, p = 200_003, 8
    ctx = zb.zg_init(n, p)
    s = zb.zg_shard_len(ctx)
    gen = torch.Generator(device="cuda").manual_seed(5)
    params = torch.randn(p * s, device="cuda", generator=gen).to(torch.bfloat16)
    codes = torch.randint(0, 256, (p * s,), dtype=torch.int32, device="cuda", generator=gen).to(torch.uint8)
    scales = torch.randint(110, 140, (p * s // 32,), dtype=torch.int32, device="cuda", generator=gen).to(torch.uint8)
    out = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    out_mx = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    out_dma = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    zb.zg_gather_params(ctx, params, 0, 16, out[:16])  # launch configurations cached before capture
    zb.zg_gather_params_mxfp8(ctx, codes, scales, 0, 16, out_mx[:16])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        zb.zg_gather_params(ctx, params, 0, 100_000, out[:100_000])
        zb.zg_gather_params(ctx, params, 100_000, n, out[100_000:])
        zb.zg_gather_params_mxfp8(ctx, codes, scales, 0, n, out_mx)
        zb.zg_gather_params_dma(ctx, params, 3, n, out_dma[:n - 3])
    hc, hs = codes.cpu().numpy(), scales.cpu().numpy()
    for k in range(2):
        if k:
            params.add_(1.0)  # the same buffers with new values
            codes.bitwise_xor_(0x11)
            hc = codes.cpu().numpy()
        out.zero_()
        out_mx.zero_()
        out_dma.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), params[:n].view(torch.int16)), k
        assert torch.equal(out_dma[:n - 3].view(torch.int16), params[3:n].view(torch.int16)), k
        want = oracle.gather_mx([hc[r * s:(r + 1) * s] for r in range(p)],
                                [hs[r * s // 32:(r + 1) * s // 32] for r in range(p)], s, 0, n)
        assert np.array_equal(to_host_u16(out_mx), want), k
