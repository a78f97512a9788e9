"""Plant one plausible mistake at a time in a copy of the oracle and check
that the pins catch it: a dropped term, a wrong sign, index or constant, a
swapped operand, a wrong rounding tie rule. The real oracle source is never
modified; each mutant is compiled from a temporary copy and its pins run in a
child process of its own (several at a time), so a mutant that crashes cannot
take the test run down.
"""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "zg_oracle.c")

MUTANTS = {
    "bias_correction_uses_beta2": ("d->b1p = now->b1p * hp->beta1;", "d->b1p = now->b1p * hp->beta2;"),
    "first_moment_skips_clip": ("float mi = b1 * m[i] + omb1 * ga;", "float mi = b1 * m[i] + omb1 * g[i];"),
    "second_moment_not_squared": ("float vi = b2 * v[i] + omb2 * (ga * ga);", "float vi = b2 * v[i] + omb2 * ga;"),
    "eps_inside_sqrt": ("float den = sqrtf(vh) + eps;", "float den = sqrtf(vh + eps);"),
    "weight_decay_dropped": ("float wi = w[i] - lrwd * w[i];", "float wi = w[i];"),
    "update_sign_flipped": ("wi = wi - lr * (mh / den);", "wi = wi + lr * (mh / den);"),
    "no_first_bias_correction": ("float mh = mi / d->bc1;", "float mh = mi;"),
    "no_second_bias_correction": ("float vh = vi / d->bc2;", "float vh = vi;"),
    "bias_correction_power_off_by_one": ("d->bc1 = (float)(1.0 - d->b1p);", "d->bc1 = (float)(1.0 - now->b1p * hp->beta1 * hp->beta1);"),
    "no_skip": ("d->found_inf = !isfinite(sumsq);", "d->found_inf = 0;"),
    "skip_still_counts_step": ("    if (d->found_inf)\n        return;\n    d->t = now->t + 1;",
                               "    if (d->found_inf) {\n        d->t = now->t + 1;\n        return;\n    }\n    d->t = now->t + 1;"),
    "sum_not_averaged": ("double denom = (double)loss_scale * (grad_average ? (double)p : 1.0);",
                         "double denom = (double)loss_scale;"),
    "rank_zero_dropped": ("for (int r = 0; r < p; ++r)\n            s = s + orc_bf16_to_f32(grads[r][i]);",
                          "for (int r = 1; r < p; ++r)\n            s = s + orc_bf16_to_f32(grads[r][i]);"),
    "clip_may_amplify": ("d->clip = (float)(q < 1.0 ? q : 1.0);", "d->clip = (float)q;"),
    "clip_uses_sumsq": ("double q = hp->max_grad_norm / (d->norm + hp->norm_eps);",
                        "double q = hp->max_grad_norm / (d->sumsq + hp->norm_eps);"),
    "square_not_taken": ("float q = g[i] * g[i];", "float q = g[i];"),
    "bf16_ties_away": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (dropped >= 0x8000u)"),
    "bf16_truncates": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (0)"),
    "e4m3_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0))", "if (frac >= 0.5)"),
    "e4m3_overflow_to_nan": ("mag = 0x7e;", "mag = 0x7f;"),
    "e4m3_bias_wrong": ("mag = (uint8_t)(((e + 7) << 3) + (r - 8));", "mag = (uint8_t)(((e + 8) << 3) + (r - 8));"),
    "e4m3_subnormal_step_wrong": ("mag = (uint8_t)round_half_even(a * 512.0);", "mag = (uint8_t)round_half_even(a * 256.0);"),
    "mx_scale_off_by_one": ("e = (k - 1) - emax_elem;", "e = k - emax_elem;"),
    "mx_scale_not_clamped": ("        if (e < -127)\n            e = -127;\n", ""),
    "mx_nan_block_not_poisoned": ("nonfinite = 1;", "nonfinite = 0;"),
    "mx_decode_bias_wrong": ("return (float)ldexp(v, (int)scale - 127);", "return (float)ldexp(v, (int)scale - 128);"),
    "mx_f32_through_bf16": ("vals[j] = (double)x[lo + j];",
                            "vals[j] = (double)orc_bf16_to_f32(orc_f32_to_bf16(x[lo + j]));"),
    "shard_not_block_aligned": ("return (s + 31) / 32 * 32;", "return s;"),
    "mx_reduce_scale_of_next_rank": ("s = s + orc_mx_decode(codes[r][i], scales[r][i / 32]);",
                                     "s = s + orc_mx_decode(codes[r][i], scales[(r + 1) % p][i / 32]);"),
    "gather_neighbour_offset": ("out[i - lo] = shards[r][k];", "out[i - lo] = shards[r][k ^ 1];"),
    "gather_from_rank_zero": ("out[i - lo] = shards[r][k];", "out[i - lo] = shards[0][k];"),
    "gather_mx_scale_of_rank_zero": ("scales[r][k / 32]", "scales[0][k / 32]"),
    "gather_mx_scale_per_64": ("scales[r][k / 32]", "scales[r][k / 64]"),
    "gather_mx_truncates": ("out[i - lo] = orc_f32_to_bf16(orc_mx_decode(codes[r][k], scales[r][k / 32]));",
                            "out[i - lo] = (uint16_t)(bits_from_f32(orc_mx_decode(codes[r][k], scales[r][k / 32])) >> 16);"),
    "norm_eps_dropped": ("double q = hp->max_grad_norm / (d->norm + hp->norm_eps);",
                         "double q = hp->max_grad_norm / d->norm;"),
    "decay_after_update": ("        float wi = w[i] - lrwd * w[i];\n        wi = wi - lr * (mh / den);",
                           "        float wi = w[i] - lr * (mh / den);\n        wi = wi - lrwd * wi;"),
    "second_moment_mixes_clip": ("float vi = b2 * v[i] + omb2 * (ga * ga);", "float vi = b2 * v[i] + omb2 * (ga * g[i]);"),
    "powers_in_binary32": ("    d->b1p = now->b1p * hp->beta1;\n    d->b2p = now->b2p * hp->beta2;",
                           "    d->b1p = (float)(now->b1p * hp->beta1);\n    d->b2p = (float)(now->b2p * hp->beta2);"),
    "params_from_old_weights": ("        w[i] = wi;\n        p[i] = orc_f32_to_bf16(wi);",
                                "        p[i] = orc_f32_to_bf16(w[i]);\n        w[i] = wi;"),
    "unscale_before_sum": ("        for (int r = 0; r < p; ++r)\n            s = s + orc_bf16_to_f32(grads[r][i]);\n        g[i - lo] = s * inv;",
                           "        for (int r = 0; r < p; ++r)\n            s = s + orc_bf16_to_f32(grads[r][i]) * inv;\n        g[i - lo] = s;"),
    "mx_amax_signed": ("        else if (fabs(vals[j]) > amax)\n            amax = fabs(vals[j]);",
                       "        else if (vals[j] > amax)\n            amax = vals[j];"),
    "mx_zero_block_scale_one": ("    if (amax == 0.0) {\n        e = -127;", "    if (amax == 0.0) {\n        e = 0;"),
    "clip_in_binary32": ("        double q = hp->max_grad_norm / (d->norm + hp->norm_eps);",
                         "        double q = (float)hp->max_grad_norm / ((float)d->norm + (float)hp->norm_eps);"),
    "mx_nan_scale_ignored": ("    if (scale == 0xff)\n        return NAN;\n", ""),
    "bias_correction_binary32_subtract": ("    d->bc1 = (float)(1.0 - d->b1p);", "    d->bc1 = 1.0f - (float)d->b1p;"),
    "found_inf_only_inf": ("    d->found_inf = !isfinite(sumsq);", "    d->found_inf = isinf(sumsq);"),
    "sharded_norm_drops_last_rank": ("    for (int r = 0; r < p; ++r)\n        ss = ss + partial[r];",
                                     "    for (int r = 0; r < p - 1; ++r)\n        ss = ss + partial[r];"),
    "sharded_norm_is_a_local_norm": ("    for (int r = 0; r < p; ++r)\n        ss = ss + partial[r];", "    ss = partial[0];"),
    "running_power_reset": ("    ctr->b1p = 1.0;\n    ctr->b2p = 1.0;\n    for (int64_t k = 0; k < t; ++k) {",
                            "    ctr->b1p = 1.0;\n    ctr->b2p = 1.0;\n    for (int64_t k = 1; k < t; ++k) {"),
}

_CHILD = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
lib = oracle.load({lib!r})
print("FAILED=" + json.dumps(oracle_pins.run_all(lib)))
"""


def _run_mutant(name: str, workdir: str) -> tuple[str, int, list | None]:
    """Compile one mutant in its own folder and run every pin on it in a child
    process; returns (name, the child's exit status, the failed pins)."""
    find, repl = MUTANTS[name]
    src = open(SRC).read()
    if src.count(find) != 1:
        return name, -1, None
    os.makedirs(workdir, exist_ok=True)
    mutant_src = os.path.join(workdir, "mutant.c")
    with open(mutant_src, "w") as f:
        f.write(src.replace(find, repl))
    lib = oracle.build(mutant_src, os.path.join(workdir, "libmutant.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = _CHILD.format(root=root, tests=os.path.join(root, "tests"), lib=lib)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    failed = None
    for line in proc.stdout.splitlines():
        if line.startswith("FAILED="):
            failed = json.loads(line[len("FAILED="):])
    return name, proc.returncode, failed


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every mutant built and run once, several child processes at a time
    (each still alone in its process, so a crash stays contained)."""
    base = tmp_path_factory.mktemp("mutants")
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        runs = ex.map(lambda n: _run_mutant(n, str(base / n)), sorted(MUTANTS))
        return {name: (rc, failed) for name, rc, failed in runs}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, outcomes):
    rc, failed = outcomes[name]
    assert not (rc == -1 and failed is None), f"mutation site for {name} not found exactly once"
    # a crash of the child also counts as caught; a clean run with no failed pin does not
    assert rc != 0 or (failed is not None and len(failed) > 0), f"mutant {name} passed every pin"
