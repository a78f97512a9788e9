"""Measured bytes against the formulas (Zero From Scratch, item 19).

The device memory a P-rank problem occupies, read from the allocator's own
counter, must equal the accounting: fp32 w, m, v = 12 * P * S bytes, bf16
params = 2 * P * S, and P bf16 gradient replicas = 2 * P * P * S, with S the
shard length the library reports. (Sizes are multiples of 512 bytes, the
allocator's granule, so the counter is exact.)"""
import pytest
import torch

from zero_sharded_mixed_flat_gb300 import accounting as acc
from zero_sharded_mixed_flat_gb300 import binding as zb

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,p", [(1 << 20, 8), (3_000_064, 4), (65_536, 16)])
def test_resident_bytes_match_the_formula(n, p):
    ctx = zb.zg_init(n, p)
    s = zb.zg_shard_len(ctx)
    total = p * s
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    w = torch.zeros(total, dtype=torch.float32, device="cuda")
    m = torch.zeros_like(w)
    v = torch.zeros_like(w)
    params = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    grads = [torch.zeros(total, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    zb.zg_bind(ctx, w, m, v, params)
    torch.cuda.synchronize()
    used = torch.cuda.memory_allocated() - before
    want = acc.resident_bytes(n, p, s)
    assert used == want["state"] + want["params"] + want["grads"], (used, want)
    # per weight: 12 + 2 + 2P bytes here, the 16 of a single rank's view
    # (item 1) plus the P - 1 other ranks' gradient replicas this GPU holds
    assert (want["state"] + want["params"]) / total == acc.bytes_per_weight() - acc.GRAD_BF16
    zb.zg_step(ctx, grads, 1024.0)
    assert zb.zg_get_info(ctx).step_t == 1
    del grads
