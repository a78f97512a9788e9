"""The oracle: a plain CPU statement of the sharded mixed-precision optimizer step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library and
its Python binding never import it, and it shares no code with them: the C
source here (``zg_oracle.c``) is compiled on its own with gcc.

The arithmetic lives in ``zg_oracle.c`` (fp32 per element, each operation
rounded separately; fp64 for the norm); this module only loads it and moves
numpy arrays in and out. ``ring.py`` simulates the ring collectives on P
in-memory ranks and ``quadratic.py`` holds the tiny model for the gradient
check. Every function cites the passage it follows (page title, then the item
of the "Zero From Scratch" outline, counted from 1 after its introduction).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zg_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# -ffp-contract=off: no fused multiply-add may merge two roundings into one.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` (the oracle, or a copy of it) into the shared library ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


class _Hparams(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_double),
        ("beta1", ctypes.c_double),
        ("beta2", ctypes.c_double),
        ("eps", ctypes.c_double),
        ("weight_decay", ctypes.c_double),
        ("max_grad_norm", ctypes.c_double),
        ("norm_eps", ctypes.c_double),
        ("grad_average", ctypes.c_int),
    ]


class _Counters(ctypes.Structure):
    _fields_ = [("t", ctypes.c_int64), ("b1p", ctypes.c_double), ("b2p", ctypes.c_double)]


class _Decision(ctypes.Structure):
    _fields_ = [
        ("sumsq", ctypes.c_double),
        ("norm", ctypes.c_double),
        ("clip", ctypes.c_float),
        ("bc1", ctypes.c_float),
        ("bc2", ctypes.c_float),
        ("found_inf", ctypes.c_int),
        ("t", ctypes.c_int64),
        ("b1p", ctypes.c_double),
        ("b2p", ctypes.c_double),
    ]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    sig = {
        "orc_shard_len": (_I64, [_I64, ctypes.c_int]),
        "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
        "orc_mx_encode": (None, [_P, _I64, _P, _P]),
        "orc_mx_encode_f32": (None, [_P, _I64, _P, _P]),
        "orc_mx_decode": (ctypes.c_float, [ctypes.c_uint8, ctypes.c_uint8]),
        "orc_inv_scale": (ctypes.c_float, [ctypes.c_float, ctypes.c_int, ctypes.c_int]),
        "orc_reduce_unscale": (None, [ctypes.c_int, _P, _I64, _I64, ctypes.c_float, _P]),
        "orc_mx_reduce_unscale": (None, [ctypes.c_int, _P, _P, _I64, _I64, ctypes.c_float, _P]),
        "orc_sumsq": (ctypes.c_double, [_P, _I64]),
        "orc_decide": (None, [_P, _P, ctypes.c_double, _P]),
        "orc_adamw": (None, [_P, _P, _P, _P, _P, _P, _P, _I64]),
        "orc_step": (ctypes.c_int, [_I64, ctypes.c_int, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P]),
        "orc_step_mx": (ctypes.c_int, [_I64, ctypes.c_int, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P]),
        "orc_step_sharded": (ctypes.c_int, [_I64, ctypes.c_int, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P]),
        "orc_counters_at": (None, [_P, _I64, _P]),
        "orc_gather": (None, [_I64, _P, _I64, _I64, _P]),
        "orc_gather_mx": (None, [_I64, _P, _P, _I64, _I64, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled oracle (building it first if needed). With ``path``,
    load that library instead (used by the tests that plant a mistake in a copy)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrays) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrays))(*[_ptr(a) for a in arrays])


@dataclass(frozen=True)
class Hparams:
    """AdamW + clip settings. The pages print none of these; the defaults are
    the common ones (lr 1e-3, betas 0.9/0.999, eps 1e-8, wd 0.01, clip 1.0)."""

    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 1.0
    norm_eps: float = 1e-6
    grad_average: int = 1

    def c(self) -> _Hparams:
        return _Hparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                        self.max_grad_norm, self.norm_eps, int(self.grad_average))


@dataclass
class Decision:
    sumsq: float
    norm: float
    clip: float
    bc1: float
    bc2: float
    found_inf: bool
    t: int


def _decision(d: _Decision) -> Decision:
    return Decision(d.sumsq, d.norm, d.clip, d.bc1, d.bc2, bool(d.found_inf), d.t)


# ---------------------------------------------------------------- formats

def shard_len(n: int, p: int, lib=None) -> int:
    """Shard length S (Zero From Scratch, item 17): ceil(N/P) rounded up to 32."""
    return int((lib or load()).orc_shard_len(n, p))


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32: the bits move to the top half."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray, lib=None) -> np.ndarray:
    """Round float32 to bf16 bit patterns, one call per element into the C oracle."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def e4m3_value(code: int, lib=None) -> float:
    return float((lib or load()).orc_e4m3_value(int(code)))


def e4m3_encode(y: float, lib=None) -> int:
    return int((lib or load()).orc_e4m3_encode(float(y)))


def mx_encode(x_bf16: np.ndarray, lib=None):
    """MXFP8-encode one rank's bf16 buffer (Zero From Scratch, item 14).
    Returns (codes uint8[n], scales uint8[ceil(n/32)])."""
    lib = lib or load()
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n = x.size
    codes = np.zeros(n, dtype=np.uint8)
    scales = np.zeros((n + 31) // 32, dtype=np.uint8)
    lib.orc_mx_encode(_ptr(x), n, _ptr(codes), _ptr(scales))
    return codes, scales


def mx_encode_f32(x: np.ndarray, lib=None):
    """MXFP8-encode float32 values (the master weights stored as MX
    parameters; Zero From Scratch, item 14). Returns (codes, scales)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.size
    codes = np.zeros(n, dtype=np.uint8)
    scales = np.zeros((n + 31) // 32, dtype=np.uint8)
    lib.orc_mx_encode_f32(_ptr(x), n, _ptr(codes), _ptr(scales))
    return codes, scales


def mx_decode(code: int, scale: int, lib=None) -> float:
    return float((lib or load()).orc_mx_decode(int(code), int(scale)))


def gather(shards, s: int, lo: int, hi: int, lib=None) -> np.ndarray:
    """Stage-three just-in-time gather of bf16 parameters [lo, hi) from the P
    rank shards (each S long) (DeepSpeed documentation review, paragraph on
    the three stages). Returns the bf16 patterns, uint16[hi - lo]."""
    lib = lib or load()
    shards = [np.ascontiguousarray(x, dtype=np.uint16) for x in shards]
    out = np.zeros(max(hi - lo, 0), dtype=np.uint16)
    lib.orc_gather(s, _ptr_array(shards), lo, hi, _ptr(out))
    return out


def gather_mx(codes, scales, s: int, lo: int, hi: int, lib=None) -> np.ndarray:
    """The gather from MXFP8 parameter shards (codes S long, scales S/32),
    decoded and rounded to bf16 (Zero From Scratch, item 14)."""
    lib = lib or load()
    codes = [np.ascontiguousarray(x, dtype=np.uint8) for x in codes]
    scales = [np.ascontiguousarray(x, dtype=np.uint8) for x in scales]
    out = np.zeros(max(hi - lo, 0), dtype=np.uint16)
    lib.orc_gather_mx(s, _ptr_array(codes), _ptr_array(scales), lo, hi, _ptr(out))
    return out


def inv_scale(loss_scale: float, p: int, grad_average: int = 1, lib=None) -> float:
    return float((lib or load()).orc_inv_scale(loss_scale, p, grad_average))


def reduce_unscale(grads, lo: int, hi: int, inv: float, lib=None) -> np.ndarray:
    """Rank-ordered fp32 sum of the P bf16 slices [lo, hi), times ``inv``."""
    lib = lib or load()
    g = np.empty(max(hi - lo, 0), dtype=np.float32)
    lib.orc_reduce_unscale(len(grads), _ptr_array(grads), lo, hi, inv, _ptr(g))
    return g


def mx_reduce_unscale(codes, scales, lo: int, hi: int, inv: float, lib=None) -> np.ndarray:
    lib = lib or load()
    g = np.empty(max(hi - lo, 0), dtype=np.float32)
    lib.orc_mx_reduce_unscale(len(codes), _ptr_array(codes), _ptr_array(scales), lo, hi, inv, _ptr(g))
    return g


def sumsq(g: np.ndarray, lib=None) -> float:
    g = np.ascontiguousarray(g, dtype=np.float32)
    return float((lib or load()).orc_sumsq(_ptr(g), g.size))


def counters_at(hp: Hparams, t: int, lib=None) -> tuple[int, float, float]:
    c = _Counters()
    (lib or load()).orc_counters_at(ctypes.byref(hp.c()), t, ctypes.byref(c))
    return c.t, c.b1p, c.b2p


# ---------------------------------------------------------------- optimizer

class OracleOptimizer:
    """The oracle's optimizer over one flat vector: fp32 w, m, v and bf16 p,
    all N long, plus the step counters. ``step`` runs one whole step."""

    def __init__(self, w0: np.ndarray, hp: Hparams = Hparams(), lib=None):
        self.lib = lib or load()
        self.hp = hp
        self._hp = hp.c()
        self.w = np.ascontiguousarray(w0, dtype=np.float32).copy()
        self.n = self.w.size
        self.m = np.zeros(self.n, dtype=np.float32)
        self.v = np.zeros(self.n, dtype=np.float32)
        self.p = np.zeros(self.n, dtype=np.uint16)
        self.ctr = _Counters(0, 1.0, 1.0)

    @property
    def t(self) -> int:
        return int(self.ctr.t)

    def set_step(self, t: int) -> None:
        self.lib.orc_counters_at(ctypes.byref(self._hp), t, ctypes.byref(self.ctr))

    def _args(self):
        return (ctypes.byref(self._hp), ctypes.byref(self.ctr), _ptr(self.w), _ptr(self.m),
                _ptr(self.v), _ptr(self.p))

    def step(self, grads, loss_scale: float, sharded: bool = False) -> Decision:
        """grads: P arrays of bf16 bit patterns (uint16), each at least N long."""
        for g in grads:
            assert g.dtype == np.uint16 and g.size >= self.n
        d = _Decision()
        fn = self.lib.orc_step_sharded if sharded else self.lib.orc_step
        rc = fn(self.n, len(grads), _ptr_array(grads), loss_scale, *self._args(), ctypes.byref(d))
        if rc < 0:
            raise MemoryError("oracle step could not allocate its scratch vector")
        return _decision(d)

    def step_mx(self, codes, scales, loss_scale: float) -> Decision:
        d = _Decision()
        rc = self.lib.orc_step_mx(self.n, len(codes), _ptr_array(codes), _ptr_array(scales),
                                  loss_scale, *self._args(), ctypes.byref(d))
        if rc < 0:
            raise MemoryError("oracle step could not allocate its scratch vector")
        return _decision(d)


# ----------------------------------------------------- pieces for sampled runs

def decide(hp: Hparams, t: int, b1p: float, b2p: float, total_sumsq: float, lib=None) -> Decision:
    """The step decision from a global sum of squares (norm, skip, clip, bias
    corrections), for runs too large to hold whole on the host."""
    lib = lib or load()
    now = _Counters(t, b1p, b2p)
    d = _Decision()
    lib.orc_decide(ctypes.byref(hp.c()), ctypes.byref(now), total_sumsq, ctypes.byref(d))
    return _decision(d), (d.t, d.b1p, d.b2p)


def adamw_range(hp: Hparams, dec: Decision, g: np.ndarray, w: np.ndarray, m: np.ndarray,
                v: np.ndarray, lib=None) -> np.ndarray:
    """AdamW on one contiguous range, in place on w, m, v; returns bf16 params."""
    lib = lib or load()
    d = _Decision(dec.sumsq, dec.norm, dec.clip, dec.bc1, dec.bc2, int(dec.found_inf), dec.t, 0.0, 0.0)
    p = np.zeros(w.size, dtype=np.uint16)
    for a in (g, w, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib.orc_adamw(ctypes.byref(hp.c()), ctypes.byref(d), _ptr(g), _ptr(w), _ptr(m), _ptr(v), _ptr(p), w.size)
    return p
