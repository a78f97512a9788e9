"""The stage-three exchange with real collectives, on CPU (gloo), world sizes 2
to 4.

DeepSpeed documentation review, paragraph on the three stages: stage three
splits the parameters as well, and each layer collects its parameters from
the ranks that own them right before it runs, dropping them afterwards.
Zero From Scratch, items 9 and 18: the third flag shards the parameters.

Each process runs the stage-two exchange of its optimizer step (reduce-scatter
by point-to-point sends and a rank-ordered sum, one scalar all-reduce, AdamW
on its own shard) but keeps only its own bf16 parameter shard: there is no
all-gather at the end of the step. A forward sweep over a layer table then
gathers each layer's flat range from the owners, every rank sending its part
of the range (possibly empty). The same sweep runs once more from parameter
shards stored as MXFP8 (codes plus the scale bytes of the blocks a part
touches), decoded by the receiver. Every rank's gathered layers must equal
the single-process oracle's gather of the single-process step's parameters.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from zero_sharded_mixed_flat_gb300 import synth

N = 5003
STEPS = 3
LAYERS = [(0, 700), (700, 2500), (2500, 2501), (2501, 2501), (2501, 4000), (4000, N)]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(world: int):
    w = synth.workload("flat65k_p4", n=N, p=world)
    return w, [synth.step_grads(w, t) for t in range(1, STEPS + 1)]


def _all_gather_bytes(piece: np.ndarray, world: int) -> list[np.ndarray]:
    """All-gather variable-length byte strings: lengths first, then the
    pieces padded to a common multiple of 4 bytes (gloo moves int32)."""
    n = torch.tensor([piece.size], dtype=torch.int64)
    lens = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(lens, n)
    lens = [int(x.item()) for x in lens]
    width = max(4, -(-max(lens) // 4) * 4)
    buf = np.zeros(width, np.uint8)
    buf[: piece.size] = piece
    out = [torch.empty(width // 4, dtype=torch.int32) for _ in range(world)]
    dist.all_gather(out, torch.from_numpy(buf.view(np.int32)))
    return [o.numpy().view(np.uint8)[:k] for o, k in zip(out, lens)]


def _worker(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        hp = oracle.Hparams()
        w, steps = _inputs(world)
        s = oracle.shard_len(N, world)
        lo, hi = min(rank * s, N), min((rank + 1) * s, N)
        w_shard = synth.init_weights(w, 0, N)[lo:hi].copy()
        m_shard = np.zeros(hi - lo, np.float32)
        v_shard = np.zeros(hi - lo, np.float32)
        t, b1p, b2p = 0, 1.0, 1.0
        p_shard = None  # this rank's bf16 parameters: the only ones it keeps
        for grads in steps:
            mine = torch.from_numpy(grads[rank].view(np.int32).copy())
            h = s // 2
            recv = [torch.empty(h, dtype=torch.int32) for _ in range(world)]
            recv[rank] = mine[rank * h:(rank + 1) * h].clone()
            ops = []
            for j in range(world):
                if j != rank:
                    ops.append(dist.isend(mine[j * h:(j + 1) * h].clone(), dst=j))
                    ops.append(dist.irecv(recv[j], src=j))
            for op in ops:
                op.wait()
            slices = [r.numpy().view(np.uint16) for r in recv]
            g = oracle.reduce_unscale(slices, 0, hi - lo, oracle.inv_scale(w.loss_scale, world, hp.grad_average))
            ss = torch.tensor([oracle.sumsq(g)], dtype=torch.float64)
            dist.all_reduce(ss)
            dec, (t2, b1p2, b2p2) = oracle.decide(hp, t, b1p, b2p, float(ss.item()))
            if not dec.found_inf:
                p_shard = oracle.adamw_range(hp, dec, g, w_shard, m_shard, v_shard)
                t, b1p, b2p = t2, b1p2, b2p2
        # MX parameter shard of this rank: codes for its elements, one scale per 32
        # (the shard starts on a block boundary, S being a multiple of 32)
        mx_codes, mx_scales = oracle.mx_encode_f32(w_shard)
        layers, layers_mx = [], []
        for a, b in LAYERS:
            oa, ob = max(a, lo), min(b, hi)  # this rank's part of the layer
            if ob < oa:
                oa = ob = lo
            parts = _all_gather_bytes(p_shard[oa - lo:ob - lo].view(np.uint8), world)
            layers.append(np.concatenate([x.view(np.uint16) for x in parts]))
            # MX: the codes of the part and the scale bytes of the blocks it touches
            blo, bhi = (oa - lo) // 32, -(-(ob - lo) // 32)
            cparts = _all_gather_bytes(mx_codes[oa - lo:ob - lo], world)
            sparts = _all_gather_bytes(mx_scales[blo:bhi] if ob > oa else mx_scales[:0], world)
            meta = torch.tensor([oa, ob], dtype=torch.int64)
            metas = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(metas, meta)
            # the receiver places each owner's pieces into an owner-shaped buffer and decodes
            cs = [np.zeros(s, np.uint8) for _ in range(world)]
            scs = [np.zeros(s // 32, np.uint8) for _ in range(world)]
            for r in range(world):
                ra, rb = (int(x) for x in metas[r])
                if rb > ra:
                    cs[r][ra - r * s:rb - r * s] = cparts[r]
                    b0 = (ra - r * s) // 32
                    scs[r][b0:b0 + sparts[r].size] = sparts[r]
            layers_mx.append(oracle.gather_mx(cs, scs, s, a, b))
            # the gathered layer is this rank's working copy: used, then released
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), t=t,
                 **{f"layer{i}": x for i, x in enumerate(layers)},
                 **{f"mx{i}": x for i, x in enumerate(layers_mx)})
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4])
def test_stage_three_over_gloo_matches_single_process(world, tmp_path):
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    w, steps = _inputs(world)
    ref = oracle.OracleOptimizer(synth.init_weights(w, 0, N), oracle.Hparams())
    for grads in steps:
        ref.step(grads, w.loss_scale)
    s = oracle.shard_len(N, world)
    shards = [np.pad(ref.p[r * s:(r + 1) * s], (0, s - ref.p[r * s:(r + 1) * s].size)) for r in range(world)]
    mx = [oracle.mx_encode_f32(ref.w[r * s:(r + 1) * s]) for r in range(world)]
    mx_c = [np.pad(c, (0, s - c.size)) for c, _ in mx]
    mx_s = [np.pad(sc, (0, s // 32 - sc.size)) for _, sc in mx]
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npz")
        assert int(got["t"]) == ref.t == STEPS
        for i, (a, b) in enumerate(LAYERS):
            want = oracle.gather(shards, s, a, b)
            assert np.array_equal(want, ref.p[a:b])
            assert got[f"layer{i}"].tobytes() == want.tobytes(), (r, i)
            assert got[f"mx{i}"].tobytes() == oracle.gather_mx(mx_c, mx_s, s, a, b).tobytes(), (r, i)
