"""Thin Python binding over libzg.so (declared in include/zg.h).

Argument marshalling only: torch tensors supply device pointers, torch
streams supply the cudaStream_t, and every step of the computation runs in
the library's CUDA kernels. Each ``zg_*`` function here calls the C function
of the same name and raises ``ZgError`` on a non-zero status.

There is no fallback: if ``libzg.so`` has not been built (``python -m
zero_sharded_mixed_flat_gb300.build``) or CUDA is unavailable, the first call
fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzg.so")

ZG_OK = 0
ZG_ERR_INVALID_ARG = -1
ZG_ERR_MISALIGNED = -2
ZG_ERR_NOT_BOUND = -3
ZG_ERR_CUDA = -4
ZG_ERR_DEVICE_TIMEOUT = -5
ZG_ERR_STALE_NORM = -6
ZG_ERR_NO_MEMORY = -7
ZG_ERR_STATE_PARTIAL = -8
ZG_VARIANT_LDG = 0
ZG_VARIANT_TMA = 1
ZG_VARIANT_STAGED = 2
ZG_VARIANT_SINGLE = 3
ZG_MAX_RANKS = 16
ZG_BUCKET_FIRST = 1
ZG_BUCKET_LAST = 2


class ZgError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where}: {detail} (status {code})")
        self.code = code


class _Hp(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
        ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
        ("max_grad_norm", ctypes.c_double), ("norm_eps", ctypes.c_double), ("grad_average", ctypes.c_int),
    ]


class _Info(ctypes.Structure):
    _fields_ = [
        ("sumsq", ctypes.c_double), ("norm", ctypes.c_double), ("clip_coef", ctypes.c_float),
        ("found_inf", ctypes.c_int), ("step_t", ctypes.c_int64), ("status", ctypes.c_int),
    ]


@dataclass(frozen=True)
class Hparams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 1.0
    norm_eps: float = 1e-6
    grad_average: int = 1


@dataclass
class StepInfo:
    sumsq: float
    norm: float
    clip_coef: float
    found_inf: bool
    step_t: int
    status: int


_lib = None
_P, _I64 = ctypes.c_void_p, ctypes.c_int64


def lib() -> ctypes.CDLL:
    """Load libzg.so from the package directory (no search path, no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m zero_sharded_mixed_flat_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "zg_init": (ctypes.c_int, [_I64, ctypes.c_int, ctypes.POINTER(_Hp), ctypes.POINTER(_P)]),
            "zg_shard_len": (_I64, [_P]),
            "zg_bind": (ctypes.c_int, [_P, _P, _P, _P, _P]),
            "zg_bind_grad_stage": (ctypes.c_int, [_P, _P]),
            "zg_bind_params_mxfp8": (ctypes.c_int, [_P, _P, _P]),
            "zg_step": (ctypes.c_int, [_P, _P, ctypes.c_float, _P]),
            "zg_grad_norm": (ctypes.c_int, [_P, _P, ctypes.c_float, _P]),
            "zg_shard_step": (ctypes.c_int, [_P, _P, ctypes.c_float, _P]),
            "zg_grad_norm_bucket": (ctypes.c_int, [_P, _P, _I64, _I64, ctypes.c_float, ctypes.c_int, _P]),
            "zg_quant_mxfp8": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
            "zg_step_mxfp8": (ctypes.c_int, [_P, _P, _P, ctypes.c_float, _P]),
            "zg_grad_norm_mxfp8": (ctypes.c_int, [_P, _P, _P, ctypes.c_float, _P]),
            "zg_shard_step_mxfp8": (ctypes.c_int, [_P, _P, _P, ctypes.c_float, _P]),
            "zg_quant_norm_mxfp8": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_float, _P]),
            "zg_get_info": (ctypes.c_int, [_P, _P, ctypes.POINTER(_Info)]),
            "zg_set_step": (ctypes.c_int, [_P, _I64, _P]),
            "zg_set_variant": (ctypes.c_int, [_P, ctypes.c_int]),
            "zg_set_wait_limit": (ctypes.c_int, [_P, _I64]),
            "zg_probe_copy": (ctypes.c_int, [_P, _P, _I64, _P]),
            "zg_gather_params": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
            "zg_gather_params_mxfp8": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _P]),
            "zg_gather_params_dma": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
            "zg_grad_norm_noalloc": (ctypes.c_int, [_P, ctypes.c_int, _I64, ctypes.c_float, ctypes.c_int, _P, _P]),
            "zg_destroy": (None, [_P]),
            "zg_strerror": (ctypes.c_char_p, [ctypes.c_int]),
            "zg_last_error": (ctypes.c_char_p, []),
            "zg_version": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != ZG_OK:
        L = lib()
        detail = (L.zg_last_error() or b"").decode() or L.zg_strerror(rc).decode()
        raise ZgError(rc, where, detail)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev_ptr(t: torch.Tensor, dtype: torch.dtype, min_numel: int, what: str, host_ok: bool = False) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a tensor")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise TypeError(f"{what} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError(f"{what} must have dtype {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{what} holds {t.numel()} elements, needs at least {min_numel}")
    return t.data_ptr()


def _ptr_array(ptrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


class Ctx:
    """Owns one zg_ctx handle; remembers N and P for the marshalling checks."""

    def __init__(self, handle: int, n: int, p: int):
        self.handle, self.n, self.p = handle, n, p

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.zg_destroy(self.handle)
            self.handle = None


# ----------------------------------------------------------------- the C ABI

def zg_init(n: int, p: int, hp: Hparams = Hparams()) -> Ctx:
    out = ctypes.c_void_p()
    h = _Hp(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm, hp.norm_eps, int(hp.grad_average))
    _check(lib().zg_init(n, p, ctypes.byref(h), ctypes.byref(out)), "zg_init")
    return Ctx(out.value, n, p)


def zg_shard_len(ctx: Ctx) -> int:
    return int(lib().zg_shard_len(ctx.handle))


def zg_bind(ctx: Ctx, w: torch.Tensor, m: torch.Tensor, v: torch.Tensor, params: torch.Tensor) -> None:
    """w, m, v may be CUDA tensors or pinned host tensors (optimizer state
    offloaded to host memory, read and written by the kernels in place)."""
    ptrs = [_dev_ptr(w, torch.float32, ctx.n, "w", True), _dev_ptr(m, torch.float32, ctx.n, "m", True),
            _dev_ptr(v, torch.float32, ctx.n, "v", True), _dev_ptr(params, torch.bfloat16, ctx.n, "params")]
    _check(lib().zg_bind(ctx.handle, *ptrs), "zg_bind")
    ctx._state = (w, m, v, params)  # keep the memory alive while bound


def zg_bind_grad_stage(ctx: Ctx, stage: torch.Tensor) -> None:
    _check(lib().zg_bind_grad_stage(ctx.handle, _dev_ptr(stage, torch.float32, ctx.n, "stage")), "zg_bind_grad_stage")
    ctx._stage = stage


def zg_bind_params_mxfp8(ctx: Ctx, codes: torch.Tensor | None, scales: torch.Tensor | None) -> None:
    """Write the parameters as MXFP8 codes + scales instead of bf16 (None, None: back to bf16)."""
    if codes is None and scales is None:
        _check(lib().zg_bind_params_mxfp8(ctx.handle, None, None), "zg_bind_params_mxfp8")
        ctx._mx_params = None
        return
    c = _dev_ptr(codes, torch.uint8, ctx.n, "codes")
    s = _dev_ptr(scales, torch.uint8, (ctx.n + 31) // 32, "scales")
    _check(lib().zg_bind_params_mxfp8(ctx.handle, c, s), "zg_bind_params_mxfp8")
    ctx._mx_params = (codes, scales)


def _grads(ctx: Ctx, grads) -> ctypes.Array:
    if len(grads) != ctx.p:
        raise ValueError(f"expected {ctx.p} gradient buffers, got {len(grads)}")
    return _ptr_array([_dev_ptr(g, torch.bfloat16, ctx.n, f"grads[{r}]") for r, g in enumerate(grads)])


def _mx(ctx: Ctx, codes, scales):
    if len(codes) != ctx.p or len(scales) != ctx.p:
        raise ValueError(f"expected {ctx.p} code and scale buffers")
    nb = (ctx.n + 31) // 32
    c = _ptr_array([_dev_ptr(x, torch.uint8, ctx.n, f"codes[{r}]") for r, x in enumerate(codes)])
    s = _ptr_array([_dev_ptr(x, torch.uint8, nb, f"scales[{r}]") for r, x in enumerate(scales)])
    return c, s


def zg_step(ctx: Ctx, grads, loss_scale: float, stream=None) -> None:
    _check(lib().zg_step(ctx.handle, _grads(ctx, grads), loss_scale, _stream(stream)), "zg_step")


def zg_grad_norm(ctx: Ctx, grads, loss_scale: float, stream=None) -> None:
    _check(lib().zg_grad_norm(ctx.handle, _grads(ctx, grads), loss_scale, _stream(stream)), "zg_grad_norm")


def zg_grad_norm_bucket(ctx: Ctx, grads, lo: int, hi: int, loss_scale: float, flags: int, stream=None) -> None:
    _check(lib().zg_grad_norm_bucket(ctx.handle, _grads(ctx, grads), lo, hi, loss_scale, flags, _stream(stream)),
           "zg_grad_norm_bucket")


def zg_shard_step(ctx: Ctx, grads, loss_scale: float, stream=None) -> None:
    _check(lib().zg_shard_step(ctx.handle, _grads(ctx, grads), loss_scale, _stream(stream)), "zg_shard_step")


def _shard_ptrs(ctx: Ctx, shards, dtype: torch.dtype, block: int, what: str) -> ctypes.Array:
    """P shard pointers, one unit per ``block`` parameters (1 for values and
    codes, 32 for MX scales): from P tensors (rank r's part), or from one
    tensor holding all P shards end to end (rank r's part starts at unit
    r * S / block; ranks that own nothing get a pointer that is never read)."""
    s = zg_shard_len(ctx)
    if isinstance(shards, torch.Tensor):
        base = _dev_ptr(shards, dtype, -(-ctx.n // block), what)
        return _ptr_array([base + r * (s // block) * shards.element_size() for r in range(ctx.p)])
    if len(shards) != ctx.p:
        raise ValueError(f"expected {ctx.p} {what} shards, got {len(shards)}")
    need = [-(-max(0, min(s, ctx.n - r * s)) // block) for r in range(ctx.p)]
    return _ptr_array([_dev_ptr(x, dtype, need[r], f"{what}[{r}]") for r, x in enumerate(shards)])


def zg_gather_params(ctx: Ctx, shards, lo: int, hi: int, out: torch.Tensor, stream=None) -> None:
    """Stage three: parameters [lo, hi) gathered from the P bf16 shards into
    out[0, hi - lo). ``shards``: P tensors, or the whole parameter vector."""
    sp = _shard_ptrs(ctx, shards, torch.bfloat16, 1, "shards")
    o = _dev_ptr(out, torch.bfloat16, max(hi - lo, 0), "out")
    _check(lib().zg_gather_params(ctx.handle, sp, lo, hi, o, _stream(stream)), "zg_gather_params")


def zg_gather_params_dma(ctx: Ctx, shards, lo: int, hi: int, out: torch.Tensor, stream=None) -> None:
    """zg_gather_params on the copy engines (one device-to-device copy per shard crossed)."""
    sp = _shard_ptrs(ctx, shards, torch.bfloat16, 1, "shards")
    o = _dev_ptr(out, torch.bfloat16, max(hi - lo, 0), "out")
    _check(lib().zg_gather_params_dma(ctx.handle, sp, lo, hi, o, _stream(stream)), "zg_gather_params_dma")


def zg_gather_params_mxfp8(ctx: Ctx, codes, scales, lo: int, hi: int, out: torch.Tensor, stream=None) -> None:
    """The gather from MXFP8 parameter shards, decoded to bf16. ``codes`` and
    ``scales``: P tensors each, or the whole code and scale vectors."""
    cp = _shard_ptrs(ctx, codes, torch.uint8, 1, "codes")
    sp = _shard_ptrs(ctx, scales, torch.uint8, 32, "scales")
    o = _dev_ptr(out, torch.bfloat16, max(hi - lo, 0), "out")
    _check(lib().zg_gather_params_mxfp8(ctx.handle, cp, sp, lo, hi, o, _stream(stream)), "zg_gather_params_mxfp8")


def zg_quant_mxfp8(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, n: int | None = None,
                   stream=None) -> None:
    n = x.numel() if n is None else n
    ptrs = (_dev_ptr(x, torch.bfloat16, n, "in"), _dev_ptr(codes, torch.uint8, n, "codes"),
            _dev_ptr(scales, torch.uint8, (n + 31) // 32, "scales"))
    _check(lib().zg_quant_mxfp8(ptrs[0], n, ptrs[1], ptrs[2], _stream(stream)), "zg_quant_mxfp8")


def zg_step_mxfp8(ctx: Ctx, codes, scales, loss_scale: float, stream=None) -> None:
    c, s = _mx(ctx, codes, scales)
    _check(lib().zg_step_mxfp8(ctx.handle, c, s, loss_scale, _stream(stream)), "zg_step_mxfp8")


def zg_grad_norm_mxfp8(ctx: Ctx, codes, scales, loss_scale: float, stream=None) -> None:
    c, s = _mx(ctx, codes, scales)
    _check(lib().zg_grad_norm_mxfp8(ctx.handle, c, s, loss_scale, _stream(stream)), "zg_grad_norm_mxfp8")


def zg_quant_norm_mxfp8(ctx: Ctx, grads, codes, scales, loss_scale: float, stream=None) -> None:
    """Encode the P bf16 gradients into ``codes``/``scales`` and take the norm
    pass from the encoded values, in one launch."""
    g = _grads(ctx, grads)
    c, s = _mx(ctx, codes, scales)
    _check(lib().zg_quant_norm_mxfp8(ctx.handle, g, c, s, loss_scale, _stream(stream)), "zg_quant_norm_mxfp8")


def zg_shard_step_mxfp8(ctx: Ctx, codes, scales, loss_scale: float, stream=None) -> None:
    c, s = _mx(ctx, codes, scales)
    _check(lib().zg_shard_step_mxfp8(ctx.handle, c, s, loss_scale, _stream(stream)), "zg_shard_step_mxfp8")


def zg_get_info(ctx: Ctx, stream=None) -> StepInfo:
    i = _Info()
    _check(lib().zg_get_info(ctx.handle, _stream(stream), ctypes.byref(i)), "zg_get_info")
    return StepInfo(i.sumsq, i.norm, i.clip_coef, bool(i.found_inf), int(i.step_t), int(i.status))


def zg_set_step(ctx: Ctx, t: int, stream=None) -> None:
    """Resume at applied-step count t, in stream order (does not wait)."""
    _check(lib().zg_set_step(ctx.handle, t, _stream(stream)), "zg_set_step")


def zg_set_variant(ctx: Ctx, variant: int) -> None:
    _check(lib().zg_set_variant(ctx.handle, variant), "zg_set_variant")


def zg_set_wait_limit(ctx: Ctx, polls: int) -> None:
    _check(lib().zg_set_wait_limit(ctx.handle, polls), "zg_set_wait_limit")


def zg_probe_copy(src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """Copy src's bytes into dst with the library's streaming copy kernel
    (both CUDA tensors, contiguous; any dtype, byte count a multiple of 16)."""
    nbytes = src.numel() * src.element_size() if isinstance(src, torch.Tensor) else 0
    s = _dev_ptr(src, src.dtype if isinstance(src, torch.Tensor) else None, 0, "src")
    d = _dev_ptr(dst, dst.dtype if isinstance(dst, torch.Tensor) else None, 0, "dst")
    if dst.numel() * dst.element_size() < nbytes:
        raise ValueError("dst smaller than src")
    _check(lib().zg_probe_copy(s, d, nbytes, _stream(stream)), "zg_probe_copy")


def zg_grad_norm_noalloc(grads, n: int, loss_scale: float, out: torch.Tensor, grad_average: int = 1,
                         stream=None) -> None:
    """The norm pass without any device allocation: writes sum of squares and
    norm into ``out`` (a CUDA float64 tensor of at least two elements)."""
    ptrs = _ptr_array([_dev_ptr(g, torch.bfloat16, n, f"grads[{r}]") for r, g in enumerate(grads)])
    o = _dev_ptr(out, torch.float64, 2, "out")
    _check(lib().zg_grad_norm_noalloc(ptrs, len(grads), n, loss_scale, grad_average, o, _stream(stream)),
           "zg_grad_norm_noalloc")


def zg_version() -> int:
    return int(lib().zg_version())


# ----------------------------------------------------------------- convenience

class ShardedAdamW:
    """A context plus torch-allocated state: fp32 w, m, v and bf16 params,
    each N long, bound to the context. With ``offload`` the fp32 state lives
    in pinned host memory and the kernels read and write it there."""

    def __init__(self, n: int, p: int, hp: Hparams = Hparams(), w0: torch.Tensor | None = None,
                 device: str | torch.device = "cuda", offload: bool = False):
        self.ctx = zg_init(n, p, hp)
        self.n, self.p, self.hp = n, p, hp

        def state(init=None):
            if offload:
                t = torch.zeros(n, dtype=torch.float32, pin_memory=True)
            else:
                t = torch.zeros(n, dtype=torch.float32, device=device)
            if init is not None:
                t.copy_(init.to(torch.float32).reshape(-1))
            return t

        self.w = state(w0)
        self.m = state()
        self.v = state()
        self.params = self.w.to(device=device, dtype=torch.bfloat16)
        zg_bind(self.ctx, self.w, self.m, self.v, self.params)

    def use_mx_params(self) -> None:
        """Store the parameters as MXFP8 (allocates codes and scales with torch)."""
        dev = self.params.device
        self.pcodes = torch.zeros(self.n, dtype=torch.uint8, device=dev)
        self.pscales = torch.zeros((self.n + 31) // 32, dtype=torch.uint8, device=dev)
        zg_bind_params_mxfp8(self.ctx, self.pcodes, self.pscales)

    def use_staged(self) -> None:
        """Switch to the staged variant (allocates the fp32 stage with torch)."""
        self.stage = torch.empty(self.n, dtype=torch.float32, device=self.w.device)
        zg_bind_grad_stage(self.ctx, self.stage)
        zg_set_variant(self.ctx, ZG_VARIANT_STAGED)

    @property
    def shard_len(self) -> int:
        return zg_shard_len(self.ctx)

    def step(self, grads, loss_scale: float, stream=None) -> None:
        zg_step(self.ctx, grads, loss_scale, stream)

    def step_mxfp8(self, codes, scales, loss_scale: float, stream=None) -> None:
        zg_step_mxfp8(self.ctx, codes, scales, loss_scale, stream)

    def info(self, stream=None) -> StepInfo:
        return zg_get_info(self.ctx, stream)

    def gather(self, lo: int, hi: int, out: torch.Tensor | None = None, stream=None,
               dma: bool = False) -> torch.Tensor:
        """Stage three: parameters [lo, hi) gathered from the P rank shards of
        the parameter vector (from the MX shards, decoded, when MX parameters
        are bound) into ``out`` (allocated when None); ``dma`` moves bf16
        shards with the copy engines instead of a kernel."""
        if out is None:
            out = torch.empty(max(hi - lo, 0), dtype=torch.bfloat16, device=self.params.device)
        if getattr(self, "pcodes", None) is not None:
            zg_gather_params_mxfp8(self.ctx, self.pcodes, self.pscales, lo, hi, out, stream)
        elif dma:
            zg_gather_params_dma(self.ctx, self.params, lo, hi, out, stream)
        else:
            zg_gather_params(self.ctx, self.params, lo, hi, out, stream)
        return out
