"""The C-ABI library without a GPU: it builds, loads, exports every function
include/zg.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from zero_sharded_mixed_flat_gb300 import binding as zb
from zero_sharded_mixed_flat_gb300 import build as zbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return zb.lib()


def declared_functions() -> list[str]:
    text = open(os.path.join(ROOT, "include", "zg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zg_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 19
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(0, -8, -1):
        assert lib.zg_strerror(code)
    assert lib.zg_strerror(-99) == b"unknown status"
    assert lib.zg_version() >= 100


def test_host_side_validation_needs_no_gpu(lib):
    hp = zb._Hp(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 1e-6, 1)
    out = ctypes.c_void_p()
    for n, p in ((0, 4), (-1, 4), (1 << 62, 4), (10, 0), (10, 17)):
        assert lib.zg_init(n, p, ctypes.byref(hp), ctypes.byref(out)) == zb.ZG_ERR_INVALID_ARG
        assert out.value is None
    for field, bad in (("beta1", 1.0), ("beta2", -0.1), ("lr", float("nan")), ("eps", -1.0), ("grad_average", 2)):
        h = zb._Hp(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 1e-6, 1)
        setattr(h, field, bad)
        assert lib.zg_init(10, 2, ctypes.byref(h), ctypes.byref(out)) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_init(10, 2, None, ctypes.byref(out)) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_shard_len(None) == -1
    assert lib.zg_step(None, None, 1.0, None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_get_info(None, None, None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_quant_mxfp8(None, -1, None, None, None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_quant_mxfp8(None, 0, None, None, None) == zb.ZG_OK  # nothing to do
    assert lib.zg_probe_copy(None, None, 15, None) == zb.ZG_ERR_INVALID_ARG
    assert b"multiple of 16" in lib.zg_last_error()
    assert lib.zg_gather_params(None, None, 0, 0, None, None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_gather_params_mxfp8(None, None, None, 0, 0, None, None) == zb.ZG_ERR_INVALID_ARG
    assert lib.zg_gather_params_dma(None, None, 0, 0, None, None) == zb.ZG_ERR_INVALID_ARG
    lib.zg_destroy(None)


def test_no_cpu_fallback_without_a_gpu(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(zb.ZgError) as e:
        zb.zg_init(1024, 4)
    assert e.value.code == zb.ZG_ERR_CUDA


def test_binding_refuses_host_tensors_before_any_call():
    """Every device-pointer argument is checked in the binding: a host tensor
    (or a non-tensor) never reaches the library as an address."""
    import torch

    host_bf16 = torch.zeros(64, dtype=torch.bfloat16)
    host_u8 = torch.zeros(64, dtype=torch.uint8)
    host_f64 = torch.zeros(2, dtype=torch.float64)
    with pytest.raises(TypeError, match="src must be a CUDA tensor"):
        zb.zg_probe_copy(torch.zeros(16), torch.zeros(16))
    with pytest.raises(TypeError, match="src must be a tensor"):
        zb.zg_probe_copy(12345, torch.zeros(16))
    with pytest.raises(TypeError, match="in must be a CUDA tensor"):
        zb.zg_quant_mxfp8(host_bf16, host_u8, host_u8)
    with pytest.raises(TypeError, match=r"grads\[0\] must be a CUDA tensor"):
        zb.zg_grad_norm_noalloc([host_bf16], 64, 1.0, host_f64)
    ctx = zb.Ctx(None, 64, 2)  # a handle is never reached: the checks come first
    with pytest.raises(TypeError, match=r"grads\[0\] must be a CUDA tensor"):
        zb.zg_step(ctx, [host_bf16, host_bf16], 1.0)
    with pytest.raises(ValueError, match="expected 2 gradient buffers"):
        zb.zg_step(ctx, [host_bf16], 1.0)
    with pytest.raises(TypeError, match="w must be a CUDA tensor or pinned host memory"):
        zb.zg_bind(ctx, torch.zeros(64), torch.zeros(64), torch.zeros(64), host_bf16)



def _header_prototypes() -> dict[str, tuple[str, int]]:
    """name -> (return type, parameter count) for every function in zg.h."""
    text = open(os.path.join(ROOT, "include", "zg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(line for line in text.splitlines() if not line.lstrip().startswith("#"))
    out = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w\s\*]*?)\b(zg_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        count = 0 if params in ("", "void") else params.count(",") + 1
        out[name] = (" ".join(ret.split()), count)
    return out


def test_binding_signatures_match_the_header(lib):
    """Every function the binding declares has the header's parameter count and
    a matching kind of return value, so the two cannot drift apart."""
    protos = _header_prototypes()
    assert set(protos) == set(declared_functions())
    for name, (ret, count) in protos.items():
        fn = getattr(lib, name)
        assert len(fn.argtypes) == count, (name, len(fn.argtypes), count)
        if ret == "void":
            assert fn.restype is None, name
        elif ret.endswith("*"):
            assert fn.restype is ctypes.c_char_p, name  # the two string getters
        elif ret == "int64_t":
            assert fn.restype is ctypes.c_int64, name
        else:
            assert ret == "int" and fn.restype is ctypes.c_int, (name, ret)


def test_struct_layouts_match_the_header(tmp_path):
    """zg_hparams and zg_step_info as the binding lays them out (ctypes) equal
    what a C compiler makes of include/zg.h: size and every field's offset."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"zg_hparams": zb._Hp, "zg_step_info": zb._Info}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "zg.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        cname, field, value = line.split()
        got[(cname, field)] = int(value)
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert got[(cname, field)] == getattr(cls, field).offset, (cname, field)


def test_plain_c_program_compiles_and_links_against_the_abi(lib, tmp_path):
    """tests/c_abi_caller.c (the C caller the GPU test runs) builds with gcc
    against include/zg.h alone and links with libzg.so and the CUDA runtime:
    the header is plain C11 and every symbol it uses resolves. It is not run
    here (that needs a GPU)."""
    import glob
    import shutil
    import subprocess

    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(zbuild.nvcc())))
    hits = [h for pat in ("lib64/libcudart.so", "targets/*/lib/libcudart.so", "lib/libcudart.so")
            for h in glob.glob(os.path.join(cuda, pat))]
    if not hits:
        pytest.skip("no CUDA runtime library to link against")
    pkg = os.path.dirname(zb.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_caller.c"),
                    "-o", str(tmp_path / "caller"), "-L", pkg, "-lzg", "-L", os.path.dirname(hits[0]), "-lcudart",
                    f"-Wl,-rpath,{pkg}"], check=True)
    assert (tmp_path / "caller").exists()
