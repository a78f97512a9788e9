"""The C ABI from a plain C program: tests/c_abi_caller.c is compiled with
gcc against include/zg.h and linked with libzg.so and the CUDA runtime alone.
It allocates its buffers with cudaMalloc, runs steps through zg_init,
zg_bind, zg_step and zg_get_info, and writes its state back; the result must
match the oracle on the same seeded inputs (one step clips)."""
import glob
import os
import subprocess

import numpy as np
import pytest

import oracle
from gpu_helpers import bf16_ulp_diff, rel_errors
from zero_sharded_mixed_flat_gb300 import build as zbuild
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_root() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(zbuild.nvcc())))


def _cudart_dir(cuda: str) -> str:
    for pattern in ("lib64/libcudart.so", "targets/*/lib/libcudart.so", "lib/libcudart.so"):
        hits = glob.glob(os.path.join(cuda, pattern))
        if hits:
            return os.path.dirname(hits[0])
    pytest.fail(f"libcudart.so not found under {cuda}")


def test_c_program_through_the_abi_matches_oracle(tmp_path):
    lib = zbuild.build()
    pkg = os.path.dirname(lib)
    cuda = _cuda_root()
    exe = tmp_path / "c_abi_caller"
    subprocess.run(["gcc", "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(HERE, "c_abi_caller.c"), "-o", str(exe), "-L", pkg, "-lzg",
                    "-L", _cudart_dir(cuda), "-lcudart", f"-Wl,-rpath,{pkg}"], check=True)

    n, p, steps, L = 10_007, 4, 3, 1024.0
    w0 = (np.random.default_rng(21).standard_normal(n) * 0.02).astype(np.float32)
    grads = [[synth.random_bf16(n, seed=4000 + 10 * t + r, scale=(1e-3 if t != 1 else 1.0) * L)
              for r in range(p)] for t in range(steps)]
    src = tmp_path / "in.bin"
    with open(src, "wb") as f:
        f.write(w0.tobytes())
        for step in grads:
            for g in step:
                f.write(g.astype(np.uint16).tobytes())
    out = tmp_path / "out.bin"
    proc = subprocess.run([str(exe), str(n), str(p), str(steps), str(L), str(src), str(out)],
                          capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr

    raw = open(out, "rb").read()
    off = 0
    state = {}
    for k, dt, size in (("w", np.float32, 4), ("m", np.float32, 4), ("v", np.float32, 4), ("p", np.uint16, 2)):
        state[k] = np.frombuffer(raw, dtype=dt, count=n, offset=off)
        off += n * size
    rec = np.dtype([("sumsq", "<f8"), ("norm", "<f8"), ("clip", "<f4"), ("found_inf", "<i4"), ("t", "<i8"),
                    ("status", "<i4")])
    infos = np.frombuffer(raw, dtype=rec, count=steps, offset=off)
    assert off + steps * rec.itemsize == len(raw)

    ref = oracle.OracleOptimizer(w0)
    clipped = False
    for t in range(steps):
        dec = ref.step(grads[t], L)
        info = infos[t]
        assert info["status"] == 0 and info["found_inf"] == dec.found_inf and info["t"] == ref.t
        assert abs(info["norm"] - dec.norm) <= 1e-5 * dec.norm
        clipped |= dec.clip < 1.0
    assert clipped
    for k in ("w", "m", "v"):
        assert rel_errors(state[k], getattr(ref, k)).max() <= 2e-6 * steps, k
    assert bf16_ulp_diff(state["p"], ref.p).max() <= 1
