"""The stage-two exchange with the MXFP8 wire, on CPU (gloo), world sizes 2
to 4.

Zero From Scratch, item 14: MXFP8 halves the gradient bytes on the wire.
Each process encodes its own rank's bf16 gradient (E4M3 codes, one E8M0 scale
per 32 elements), sends every other rank the codes and scale bytes of that
rank's shard (point to point), decodes and sums the P received shards in rank
order, takes one scalar all-reduce of the sum of squares, updates its own
shard with AdamW and all-gathers the bf16 parameters. Every rank must end
with the single-process oracle's MX step bit for bit, and the bytes each rank
sends must be (P - 1) / P of its encoded payload: about half of what the bf16
exchange sends.
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

N = 6007
STEPS = 3


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(world: int):
    w = synth.workload("mxfp8_128m_p8", n=N, p=world)
    return w, [synth.step_grads(w, t) for t in range(1, STEPS + 1)]


def _exchange(mine: np.ndarray, world: int, rank: int, s_units: int) -> list[np.ndarray]:
    """All-to-all of byte shards: rank j receives unit range [j*s, (j+1)*s)
    of every rank's buffer (as int32 words, gloo's type)."""
    words = torch.from_numpy(np.ascontiguousarray(mine).view(np.int32).copy())
    h = s_units // 4
    recv = [torch.empty(h, dtype=torch.int32) for _ in range(world)]
    recv[rank] = words[rank * h:(rank + 1) * h].clone()
    ops = []
    for j in range(world):
        if j != rank:
            ops.append(dist.isend(words[j * h:(j + 1) * h].clone(), dst=j))
            ops.append(dist.irecv(recv[j], src=j))
    for op in ops:
        op.wait()
    return [r.numpy().view(np.uint8) for r in recv]


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
        sent = 0
        params = None
        for grads in steps:
            # this rank encodes its whole (padded) gradient buffer, P * S long
            codes, scales = oracle.mx_encode(grads[rank])
            # S is a multiple of 32: shard j's codes are S bytes, its scales S / 32 bytes;
            # pad the scale buffer so every shard is a whole number of int32 words
            sc_units = -(-(s // 32) // 4) * 4
            sc_pad = np.zeros(world * sc_units, np.uint8)
            for j in range(world):
                sc_pad[j * sc_units:j * sc_units + s // 32] = scales[j * (s // 32):(j + 1) * (s // 32)]
            got_c = _exchange(codes, world, rank, s)
            got_s = [x[:s // 32] for x in _exchange(sc_pad, world, rank, sc_units)]
            sent += (world - 1) * (s + s // 32)
            inv = oracle.inv_scale(w.loss_scale, world, hp.grad_average)
            g = oracle.mx_reduce_unscale(got_c, got_s, 0, hi - lo, inv)  # decode, rank-ordered sum
            ss = torch.tensor([oracle.sumsq(g)], dtype=torch.float64)
            dist.all_reduce(ss)
            dec, (t2, b1p2, b2p2) = oracle.decide(hp, t, b1p, b2p, float(ss.item()))
            if not dec.found_inf:
                p_shard = oracle.adamw_range(hp, dec, g, w_shard, m_shard, v_shard)
                t, b1p, b2p = t2, b1p2, b2p2
                padded = np.zeros(s, np.uint16)
                padded[: hi - lo] = p_shard
                gathered = [torch.empty(s // 2, dtype=torch.int32) for _ in range(world)]
                dist.all_gather(gathered, torch.from_numpy(padded.view(np.int32)))
                params = np.concatenate([x.numpy().view(np.uint16) for x in gathered])[:N]
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), w=w_shard, m=m_shard, v=v_shard, p=params, t=t,
                 lo=lo, hi=hi, sent=sent)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4])
def test_mx_wire_exchange_over_gloo_matches_single_process(world, tmp_path):
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    w, steps = _inputs(world)
    ref = oracle.OracleOptimizer(synth.init_weights(w, 0, N), oracle.Hparams())
    s = oracle.shard_len(N, world)
    for grads in steps:
        enc = [oracle.mx_encode(g) for g in grads]
        ref.step_mx([c for c, _ in enc], [sc for _, sc in enc], w.loss_scale)
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npz")
        lo, hi = int(got["lo"]), int(got["hi"])
        assert int(got["t"]) == ref.t == STEPS
        assert got["w"].tobytes() == ref.w[lo:hi].tobytes()
        assert got["m"].tobytes() == ref.m[lo:hi].tobytes()
        assert got["v"].tobytes() == ref.v[lo:hi].tobytes()
        assert got["p"].tobytes() == ref.p.tobytes()
        # MXFP8 on the wire: (P - 1) shards of S codes + S/32 scales per step,
        # against (P - 1) shards of 2 S bytes for bf16
        assert int(got["sent"]) == STEPS * (world - 1) * (s + s // 32)
        assert int(got["sent"]) / (STEPS * (world - 1) * 2 * s) == pytest.approx((1 + 1 / 32) / 2)
