"""The stage-two exchange with real collectives, on CPU, world sizes 2 to 4 (gloo).

DeepSpeed documentation review, paragraph on the stages: stage two shards the
optimizer state and the gradients. Zero From Scratch, item 7: a reduce-scatter
gives each rank the summed gradient of its own shard, and an all-gather then
hands every rank the full updated parameters; item 19: the sharded run learns
exactly what the unsharded one does.

Each process holds its own rank's bf16 gradient buffer. The reduce-scatter is
an all-to-all of the shards followed by a local sum in rank order (the order
the single-process step uses), the global norm is one scalar all-reduce, each
rank updates only its shard with the oracle, and the bf16 shards are
all-gathered. The result must equal the single-process oracle bit for bit,
also with a ragged last shard (three ranks) and with a rank that owns no
parameters at all (four ranks over N = 70: S = 32, the last shard is empty).
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

STEPS = 4


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(n: int, world: int):
    w = synth.workload("flat65k_p4", n=n, p=world)
    return w, [synth.step_grads(w, t) for t in range(1, STEPS + 1)]


def _worker(rank: int, world: int, n: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        hp = oracle.Hparams()
        w, steps = _inputs(n, world)
        s = oracle.shard_len(n, world)
        lo, hi = min(rank * s, n), min((rank + 1) * s, n)
        w_shard = synth.init_weights(w, 0, n)[lo:hi].copy()
        m_shard = np.zeros(hi - lo, np.float32)
        v_shard = np.zeros(hi - lo, np.float32)
        t, b1p, b2p = 0, 1.0, 1.0
        params = None
        for grads in steps:
            # the bf16 payload travels as pairs packed in int32 words (S is even)
            mine = torch.from_numpy(grads[rank].view(np.int32).copy())
            h = s // 2
            # reduce-scatter, part 1: every rank sends shard j of its buffer to rank j
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
            inv = oracle.inv_scale(w.loss_scale, world, hp.grad_average)
            g = oracle.reduce_unscale(slices, 0, hi - lo, inv)  # part 2: rank-ordered sum
            ss = torch.tensor([oracle.sumsq(g)], dtype=torch.float64)
            dist.all_reduce(ss)  # the one scalar all-reduce of the step
            dec, (t2, b1p2, b2p2) = oracle.decide(hp, t, b1p, b2p, float(ss.item()))
            if not dec.found_inf:
                p_shard = oracle.adamw_range(hp, dec, g, w_shard, m_shard, v_shard)
                t, b1p, b2p = t2, b1p2, b2p2
                padded = np.zeros(s, np.uint16)
                padded[: hi - lo] = p_shard
                gathered = [torch.empty(s // 2, dtype=torch.int32) for _ in range(world)]
                dist.all_gather(gathered, torch.from_numpy(padded.view(np.int32)))
                params = np.concatenate([x.numpy().view(np.uint16) for x in gathered])[:n]
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), w=w_shard, m=m_shard, v=v_shard,
                 p=params, t=t, lo=lo, hi=hi)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n", [(2, 5003), (3, 5003), (4, 70)])
def test_stage_two_over_gloo_matches_single_process(world, n, tmp_path):
    mp.start_processes(_worker, args=(world, n, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    w, steps = _inputs(n, world)
    ref = oracle.OracleOptimizer(synth.init_weights(w, 0, n), oracle.Hparams())
    for grads in steps:
        ref.step(grads, w.loss_scale)
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npz")
        lo, hi = int(got["lo"]), int(got["hi"])
        assert int(got["t"]) == ref.t == STEPS
        assert got["w"].tobytes() == ref.w[lo:hi].tobytes()
        assert got["m"].tobytes() == ref.m[lo:hi].tobytes()
        assert got["v"].tobytes() == ref.v[lo:hi].tobytes()
        assert got["p"].tobytes() == ref.p.tobytes()  # every rank holds all params after the gather
    if n == 70:
        assert (int(got["lo"]), int(got["hi"])) == (70, 70)  # the last rank owned nothing
