"""The seeded input generator: reproducible, slice-independent, right shape."""
import numpy as np

from zero_sharded_mixed_flat_gb300 import synth


def test_slices_are_independent_of_the_request():
    w = synth.workload("flat16m_p8")
    whole = synth.grads_bf16(w, 3, 5, 0, 3 * synth.CHUNK + 77)
    part = synth.grads_bf16(w, 3, 5, synth.CHUNK - 10, 2 * synth.CHUNK + 5)
    assert np.array_equal(part, whole[synth.CHUNK - 10:2 * synth.CHUNK + 5])
    again = synth.grads_bf16(w, 3, 5, 0, 3 * synth.CHUNK + 77)
    assert np.array_equal(whole, again)
    other = synth.grads_bf16(w, 3, 6, 0, 1000)
    assert not np.array_equal(other, whole[:1000])


def test_padding_and_inf_injection():
    w = synth.workload("flat16m_p8", n=10_000)
    total = synth.padded_len(w)
    assert total % (8 * 32) == 0 and total >= w.n
    k = synth.inf_index(w, w.inf_step)
    assert 0 <= k < w.n
    g = synth.grads_bf16(w, w.inf_step, w.inf_rank, 0, total)
    assert g[k] == 0x7F80 and np.all(g[w.n:] == 0)
    assert synth.inf_index(w, w.inf_step + 1) is None
    assert not np.any(synth.grads_bf16(w, w.inf_step, 0, 0, total) == 0x7F80)


def test_distributions():
    w = synth.workload("flat65k_p4")
    x = synth.grad_values(w, 1, 0)
    assert abs(x.std() - 1e-3) < 2e-5 and abs(x.mean()) < 2e-5
    w0 = synth.init_weights(w)
    assert abs(w0.std() - 0.02) < 5e-4
    t = synth.grad_values(synth.workload("mxfp8_128m_p8"), 1, 0, 0, 1 << 20)
    # Student-t with 3 degrees of freedom: heavy tails, median |x| ~ 0.765 * scale
    assert abs(np.median(np.abs(t)) / 1e-3 - 0.765) < 0.01
    assert np.max(np.abs(t)) > 50e-3
    sig = synth.tensor_sigmas(synth.workload("gpt2small_p8"), 1)
    assert sig.size == 148 and sig.min() >= 1e-5 and sig.max() <= 1e-2


def test_gpt2_small_layout():
    t = synth.gpt2_small_tensors()
    assert len(t) == 148 and sum(s for _, s in t) == 124_439_808
    b = synth.buckets(124_439_808)
    assert len(b) == 5 and b[-1] == (100_000_000, 124_439_808)


def test_generation_into_a_caller_buffer():
    """``out=`` fills a caller's array (a row of pinned host memory, say) with
    exactly the bits a fresh draw returns, and refuses a wrong shape or type."""
    import pytest

    w = synth.workload("flat16m_p8", n=3 * synth.CHUNK + 5)
    total = synth.padded_len(w)
    rows = np.zeros((2, total), dtype=np.uint16)
    for r in range(2):
        row = rows[r]
        assert synth.grads_bf16(w, 1, r, 0, total, out=row) is row
        assert np.array_equal(rows[r], synth.grads_bf16(w, 1, r, 0, total))
    wf = np.empty(1000, np.float32)
    synth.init_weights(w, 7, 1007, out=wf)
    assert np.array_equal(wf, synth.init_weights(w, 7, 1007))
    with pytest.raises(ValueError):
        synth.grads_bf16(w, 1, 0, 0, 100, out=np.zeros(99, np.uint16))
    with pytest.raises(ValueError):
        synth.grads_bf16(w, 1, 0, 0, 100, out=np.zeros(100, np.int16))
