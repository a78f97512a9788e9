"""Build libzg.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles on its own thread, then one nvcc call
links them into ``zero_sharded_mixed_flat_gb300/libzg.so``. No cmake, no
torch extension machinery: the library is a plain C-ABI shared object.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzg.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
    # IEEE division and square root, denormals kept: the step is defined with
    # correctly rounded binary32 operations.
    "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzg.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra: list[str] | None = None, out_lib: str = LIB, obj_dir: str = OBJ) -> str:
    """Compile every .cu under csrc/ and link ``out_lib``. ``extra`` adds nvcc
    flags (for instance -D tuning knobs); use a separate ``obj_dir`` then."""
    os.makedirs(obj_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "zg.h"))
    flags = NVCC_FLAGS + (extra or [])
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src).replace(".cu", ".o"))
        if _stale(obj, [src, *headers, __file__]):
            cmd = [cc, *flags, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            subprocess.run(cmd, check=True)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if _stale(out_lib, objs):
        tmp = out_lib + f".tmp{os.getpid()}"
        subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
