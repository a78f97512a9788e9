"""Plant one plausible mistake at a time in a copy of the ring collectives
(oracle/ring.py) and check that the ring tests catch it: a chunk index off
by one, the wrong chunk returned, an overwrite instead of an add, one hop
short, a miscounted hop or message. The real module is never modified; each
copy is loaded as a module of its own and the ring tests run against it."""
import sys
import types

import pytest

import test_collectives_and_accounting as ring_tests
from oracle import ring

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


def _load(name: str, find: str, repl: str) -> types.ModuleType:
    src = open(ring.__file__).read()
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


def test_ring_tests_pass_on_the_real_module(monkeypatch):
    """The harness itself: an unmodified copy passes every ring test."""
    monkeypatch.setattr(ring_tests, "ring", _load("identity", "import numpy as np", "import numpy as np"))
    for p in range(1, 9):
        ring_tests.test_ring_all_reduce_identity(p)
    for p in (1, 2, 3, 4, 8):
        ring_tests.test_ring_shard_equals_oracle_reduce(p)
