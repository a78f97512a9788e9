"""zg_step captured in a CUDA graph and replayed: a step makes no host round
trip and allocates nothing once its launch configuration is cached, so a
graph of steps must replay to the same bits as the same steps run eagerly,
including the device-side skip decision and the step count."""
import numpy as np
import pytest
import torch

from gpu_helpers import to_dev_bf16
from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu
L = 1024.0


@pytest.mark.parametrize("variant", ["ldg", "staged"])
def test_graph_replay_matches_eager(variant):
    n, p, steps_per_graph, replays = 65_549, 4, 3, 4
    w0 = torch.from_numpy((np.random.default_rng(4).standard_normal(n) * 0.02).astype(np.float32))
    host = [synth.random_bf16(n, seed=20 + r, scale=0.2 * L) for r in range(p)]
    bad = [h.copy() for h in host]
    bad[1][17] = 0x7F80  # a gradient set whose step must be skipped

    def make():
        opt = zb.ShardedAdamW(n, p, zb.Hparams(), w0)
        if variant == "staged":
            opt.use_staged()
        return opt

    eager, graphed = make(), make()
    dev = [to_dev_bf16(h) for h in host]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):  # warm-up: launch configurations get cached
            graphed.step(dev, L, s)
            eager.step(dev, L, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(steps_per_graph):
            graphed.step(dev, L)
    for _ in range(replays):
        g.replay()
        for _ in range(steps_per_graph):
            eager.step(dev, L)
    torch.cuda.synchronize()
    # a skipped step inside the graph: swap in the bad gradients and replay
    for d, h in zip(dev, bad):
        d.copy_(torch.from_numpy(h.view(np.int16)).view(torch.bfloat16))
    g.replay()
    for _ in range(steps_per_graph):
        eager.step(dev, L)
    torch.cuda.synchronize()
    a, b = graphed.info(), eager.info()
    assert a.step_t == b.step_t == 2 + steps_per_graph * replays and a.found_inf and b.found_inf
    for x, y in ((graphed.w, eager.w), (graphed.m, eager.m), (graphed.v, eager.v)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(graphed.params.view(torch.int16), eager.params.view(torch.int16))
