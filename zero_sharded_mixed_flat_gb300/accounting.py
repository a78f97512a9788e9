"""Byte accounting for the sharded mixed-precision step.

Zero From Scratch, item 1: one weight costs sixteen bytes, not two, when an
adaptive optimizer trains in mixed precision; the DeepSpeed documentation
review (paragraph on memory) names the parts: the gradient, two moment
estimates and a higher-precision master copy besides the weight itself. The
split used here: bf16 parameter 2 + bf16 gradient 2 + fp32 master 4 + fp32 m 4
+ fp32 v 4.

Zero From Scratch, items 9 and 18: the stages shard one class of state at a
time, and three flags (shard optimizer state, shard gradients, shard
parameters) describe every arrangement; each flag that is set divides its
class by P. Items 7, 8 and 17: collectives at ring cost. Item 14: MXFP8 stores
one byte per element plus one scale byte per 32. Item 3: an unfused chain of
elementwise operations reads and writes memory once per operation.

These formulas are also what the benchmark divides by to turn a kernel time
into bandwidth: the algorithmic bytes each kernel must move.
"""
from __future__ import annotations

from dataclasses import dataclass

PARAM_BF16 = 2
GRAD_BF16 = 2
MASTER_FP32 = 4
MOMENT_FP32 = 4  # each of m and v
OPTIMIZER_STATE = MASTER_FP32 + 2 * MOMENT_FP32  # 12
MX_BLOCK = 32
MX_BYTES_PER_ELEMENT = 1 + 1 / MX_BLOCK  # E4M3 code + share of one E8M0 scale


def bytes_per_weight() -> int:
    return PARAM_BF16 + GRAD_BF16 + OPTIMIZER_STATE


@dataclass(frozen=True)
class Stage:
    """The three flags."""

    shard_optimizer_state: bool = False
    shard_gradients: bool = False
    shard_parameters: bool = False


STAGES = {
    0: Stage(),
    1: Stage(True),
    2: Stage(True, True),
    3: Stage(True, True, True),
}


def per_gpu_bytes(n_params: int, p: int, stage: Stage) -> float:
    """Model-state bytes one GPU holds for ``n_params`` weights over P ranks."""
    params = PARAM_BF16 / (p if stage.shard_parameters else 1)
    grads = GRAD_BF16 / (p if stage.shard_gradients else 1)
    state = OPTIMIZER_STATE / (p if stage.shard_optimizer_state else 1)
    return n_params * (params + grads + state)


def replicated_floor_bytes(n_params: int, stage: Stage) -> float:
    """What stays on every GPU however large P grows: the unsharded classes."""
    return n_params * ((0 if stage.shard_parameters else PARAM_BF16)
                       + (0 if stage.shard_gradients else GRAD_BF16)
                       + (0 if stage.shard_optimizer_state else OPTIMIZER_STATE))


def ring_hops(p: int, op: str) -> int:
    """Communication rounds of a ring collective over P ranks."""
    return {"reduce_scatter": p - 1, "all_gather": p - 1, "all_reduce": 2 * (p - 1)}[op]


def ring_bytes_sent_per_rank(message_bytes: float, p: int, op: str) -> float:
    """Bytes each rank sends in a ring collective on an M-byte vector."""
    one = (p - 1) / p * message_bytes
    return {"reduce_scatter": one, "all_gather": one, "all_reduce": 2 * one}[op]


def mxfp8_stored_state_saving() -> float:
    """Fraction of the 16 B/weight saved by storing bf16 params and grads as MXFP8."""
    return 2 * (PARAM_BF16 - MX_BYTES_PER_ELEMENT) / bytes_per_weight()


def mxfp8_wire_saving() -> float:
    """Fraction of the bf16 gradient payload saved on the wire by MXFP8."""
    return (GRAD_BF16 - MX_BYTES_PER_ELEMENT) / GRAD_BF16


def unfused_memory_trips(n_ops: int) -> int:
    """Memory trips of a chain of n elementwise ops run one kernel each."""
    return 2 * n_ops


def fused_memory_trips(n_ops: int) -> int:
    return 2 if n_ops > 0 else 0


# ---- algorithmic bytes per parameter of each kernel (what a launch must move)

def shard_step_bytes_per_param(p: int) -> int:
    """Fused step: P bf16 gradient reads, fp32 w/m/v read and written, bf16 p written."""
    return GRAD_BF16 * p + 2 * OPTIMIZER_STATE + PARAM_BF16


def grad_norm_bytes_per_param(p: int) -> int:
    """Norm pass: P bf16 gradient reads."""
    return GRAD_BF16 * p


def step_bytes_per_param(p: int) -> int:
    """Whole step: the norm pass plus the fused step."""
    return grad_norm_bytes_per_param(p) + shard_step_bytes_per_param(p)


def staged_grad_norm_bytes_per_param(p: int) -> int:
    """Norm pass that also stores the reduced fp32 gradient: P bf16 reads + 4."""
    return GRAD_BF16 * p + 4


def staged_shard_step_bytes_per_param() -> int:
    """Step from the stored fp32 gradient: 4 read + state read/write + bf16 p."""
    return 4 + 2 * OPTIMIZER_STATE + PARAM_BF16


def mx_params_shard_step_bytes_per_param(p: int) -> float:
    """Fused step writing MXFP8 parameters (code + scale share) instead of bf16."""
    return GRAD_BF16 * p + 2 * OPTIMIZER_STATE + MX_BYTES_PER_ELEMENT


def mx_quant_bytes_per_param() -> float:
    """Encoding one rank's bf16 gradient: bf16 read, code + scale share written."""
    return GRAD_BF16 + MX_BYTES_PER_ELEMENT


def mx_grad_norm_bytes_per_param(p: int) -> float:
    return MX_BYTES_PER_ELEMENT * p


def mx_quant_norm_bytes_per_param(p: int) -> float:
    """Every rank encoded and the norm taken in one pass: P bf16 reads, P code
    + scale shares written (the norm reads nothing more)."""
    return p * mx_quant_bytes_per_param()


def mx_staged_quant_norm_bytes_per_param(p: int) -> float:
    """The same pass storing the reduced fp32 gradient as well."""
    return p * mx_quant_bytes_per_param() + 4


def mx_staged_grad_norm_bytes_per_param(p: int) -> float:
    """MX norm pass that also stores the reduced fp32 gradient."""
    return MX_BYTES_PER_ELEMENT * p + 4


def mx_shard_step_bytes_per_param(p: int) -> float:
    return MX_BYTES_PER_ELEMENT * p + 2 * OPTIMIZER_STATE + PARAM_BF16


def gather_bytes_per_param() -> int:
    """Stage three's gather of one bf16 parameter: read from its shard, written out."""
    return PARAM_BF16 + PARAM_BF16


def mx_gather_bytes_per_param() -> float:
    """The gather from MXFP8 shards: code + scale share read, bf16 written."""
    return MX_BYTES_PER_ELEMENT + PARAM_BF16


def resident_bytes(n_params: int, p: int, shard_len: int) -> dict:
    """Device bytes the single-GPU simulation of P ranks holds: fp32 w/m/v and
    bf16 params over P*S elements, and P bf16 gradient buffers of P*S each."""
    total = p * shard_len
    return {
        "state": 3 * MASTER_FP32 * total,
        "params": PARAM_BF16 * total,
        "grads": GRAD_BF16 * p * total,
    }
