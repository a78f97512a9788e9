"""Plant one plausible mistake at a time in a copy of the oracle's Python
parts and check that their tests catch it. Ring collectives (oracle/ring.py):
a chunk index off by one, the wrong chunk returned, an overwrite instead of an
add, one hop short, a miscounted hop or message. Quadratic model
(oracle/quadratic.py): a gradient without the 1/B, with the wrong sign or
without the transpose, central differences over h instead of 2h, a
data-parallel split with overlapping parts, ranks returning summed instead of
mean gradients. The real modules are never modified; each copy is loaded as a
module of its own and the tests run against it."""
import sys
import types

import pytest

import test_collectives_and_accounting as ring_tests
from oracle import quadratic, ring

MUTANTS = {
    "rs_chunk_off_by_one": ("            c = (r - h - 1) % p\n            msgs.append((r, (r + 1) % p, c,",
                            "            c = (r - h) % p\n            msgs.append((r, (r + 1) % p, c,"),
    "ag_chunk_off_by_one": ("            c = (r - h) % p\n            msgs.append(((r + 1) % p, c,",
                            "            c = (r - h - 1) % p\n            msgs.append(((r + 1) % p, c,"),
    "rs_returns_next_chunk": ("    return [partial[r][r] for r in range(p)]",
                              "    return [partial[r][(r + 1) % p] for r in range(p)]"),
    "rs_overwrites": ("partial[dst][c] = data + partial[dst][c]", "partial[dst][c] = data"),
    "rs_one_hop_short": ("    partial = [[xs[r][lo:hi].copy() for (lo, hi) in bounds] for r in range(p)]\n    for h in range(p - 1):",
                         "    partial = [[xs[r][lo:hi].copy() for (lo, hi) in bounds] for r in range(p)]\n    for h in range(p - 2):"),
    "rs_hop_per_message": ("            wire.send(r, partial[r][c].size)\n",
                           "            wire.send(r, partial[r][c].size)\n            wire.hops += 1\n"),
    "ag_messages_not_counted": ("            wire.send(r, have[r][c].size)\n", ""),
}


def _load(name: str, find: str, repl: str, base=ring) -> types.ModuleType:
    src = open(base.__file__).read()
    assert src.count(find) == 1, f"mutation site for {name} not found exactly once"
    modname = f"_ring_mutant_{name}"
    mod = types.ModuleType(modname)
    sys.modules[modname] = mod  # dataclasses look their module up by name
    exec(compile(src.replace(find, repl), modname, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_ring_mutant_is_caught(name, monkeypatch):
    mutant = _load(name, *MUTANTS[name])
    monkeypatch.setattr(ring_tests, "ring", mutant)
    failures = 0
    for p in range(1, 9):
        try:
            ring_tests.test_ring_all_reduce_identity(p)
        except Exception:
            failures += 1
    for p in (1, 2, 3, 4, 8):
        try:
            ring_tests.test_ring_shard_equals_oracle_reduce(p)
        except Exception:
            failures += 1
    sys.modules.pop(f"_ring_mutant_{name}", None)
    assert failures > 0, f"ring mutant {name} passed every ring test"


QUAD_MUTANTS = {
    "grad_without_mean": ('    return np.einsum("bkn,bk->n", a, r) / a.shape[0]', '    return np.einsum("bkn,bk->n", a, r)'),
    "grad_wrong_sign": ('    r = np.einsum("bkn,n->bk", a, w) - y\n    return np.einsum',
                        '    r = y - np.einsum("bkn,n->bk", a, w)\n    return np.einsum'),
    "grad_without_transpose": ('np.einsum("bkn,bk->n", a, r)', 'np.einsum("bkn,bk->n", a, r[:, ::-1])'),
    "fd_over_h": ("        g[i] = (loss(w + e, a, y) - loss(w - e, a, y)) / (2.0 * h)",
                  "        g[i] = (loss(w + e, a, y) - loss(w - e, a, y)) / h"),
    "dp_parts_overlap": ("a[r * part:(r + 1) * part], y[r * part:(r + 1) * part]",
                         "a[r * part // 2:(r + 1) * part], y[r * part // 2:(r + 1) * part]"),
    "dp_rank_sums": ("    return [grad(w, a[r * part:(r + 1) * part], y[r * part:(r + 1) * part]) for r in range(p)]",
                     "    return [grad(w, a[r * part:(r + 1) * part], y[r * part:(r + 1) * part]) * part for r in range(p)]"),
}


@pytest.mark.parametrize("name", sorted(QUAD_MUTANTS))
def test_quadratic_mutant_is_caught(name, monkeypatch):
    mutant = _load("q_" + name, *QUAD_MUTANTS[name], base=quadratic)
    monkeypatch.setattr(ring_tests, "quadratic", mutant)
    failures = 0
    try:
        ring_tests.test_finite_difference_gradient_check()
    except Exception:
        failures += 1
    for p in (1, 2, 4, 8):
        try:
            ring_tests.test_data_parallel_average_matches_single_device(p)
        except Exception:
            failures += 1
    sys.modules.pop(f"_ring_mutant_q_{name}", None)
    assert failures > 0, f"quadratic mutant {name} passed the gradient and data-parallel tests"


def test_ring_tests_pass_on_the_real_module(monkeypatch):
    """The harness itself: unmodified copies pass every test."""
    monkeypatch.setattr(ring_tests, "ring", _load("identity", "import numpy as np", "import numpy as np"))
    for p in range(1, 9):
        ring_tests.test_ring_all_reduce_identity(p)
    for p in (1, 2, 3, 4, 8):
        ring_tests.test_ring_shard_equals_oracle_reduce(p)
    monkeypatch.setattr(ring_tests, "quadratic", _load("q_identity", "import numpy as np", "import numpy as np",
                                                       base=quadratic))
    ring_tests.test_finite_difference_gradient_check()
    for p in (1, 2, 4, 8):
        ring_tests.test_data_parallel_average_matches_single_device(p)
