"""bench.py's own arm on the GPU, on small workloads: one JSON line with every
key of the benchmark contract, each holding what it claims (the roofline
fraction is achieved / peak on the step pass's mean over at least 20 timed
launches, the e2e byte counts are the bytes the step's inputs and the scalar
block occupy, the launch count is the passes per step times the timed
steps), and the per-workload sub-results of the default run."""
import io
import json
from contextlib import redirect_stdout

import pytest

import bench
from zero_sharded_mixed_flat_gb300 import synth

pytestmark = pytest.mark.gpu

K, W = 30, 3


def _line(argv: list[str]) -> dict:
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(argv) == 0
    lines = [x for x in buf.getvalue().splitlines() if x.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,n", [("flat65k_p4", None), ("mxfp8_128m_p8", 65_536)])
def test_bench_line_keeps_the_contract(workload, n):
    argv = ["--steps", str(K), "--warmup", str(W), "--workload", workload, "--no-configs"] + \
        (["--n", str(n)] if n else [])
    line = _line(argv)
    wl = synth.workload(workload, **({"n": n} if n else {}))
    total = synth.padded_len(wl)

    assert line["metric"] == bench.METRIC and line["unit"] == "params/s" and line["value"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == K and line["warmup"] == W
    assert line["ms_per_step"] == pytest.approx(wl.n * K / line["value"] * 1e3 / K, rel=1e-9)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["dtype"] == "f32" and "synthetic" in line["data"]
    assert line["config"]["workload"].startswith(workload) and line["config"]["N"] == wl.n

    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["achieved"] > 0 and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-12)
    assert roof["traffic"] is None or roof["traffic"] > 0
    assert roof["bytes_per_param"] * wl.n == pytest.approx(roof["algorithmic_bytes_per_launch"])
    assert roof["launches_timed"] >= bench.MIN_PASS_SAMPLES

    kern = line["kernels"]
    for name in ("norm", "step"):
        st = kern[name]
        assert st["launches"] >= bench.MIN_PASS_SAMPLES
        assert 0 < st["min_us"] <= st["median_us"] <= st["max_us"] and st["stdev_us"] >= 0
        assert st["min_us"] <= st["mean_us"] <= st["max_us"]
        assert st["gbs"] == pytest.approx(st["algorithmic_bytes"] / (st["mean_us"] / 1e6) / 1e9, rel=1e-9)
    assert roof["achieved"] == kern["step"]["gbs"] and roof["duration_us"] == kern["step"]["mean_us"]
    assert kern["passes_sum_us"] == pytest.approx(sum(kern[k]["mean_us"] for k in ("norm", "step", "encode")
                                                      if k in kern))
    assert kern["whole_step_us"] == pytest.approx(line["ms_per_step"] * 1e3)

    e2e = line["e2e"]
    assert e2e["unit"] == "params/s" and e2e["value"] > 0 and e2e["serial"] > 0
    # inputs copied every step: the P bf16 buffers, or the P ranks' codes and scales
    want_in = wl.p * total * 2 if not wl.mx else wl.p * (total + total // 32)
    assert e2e["h2d_bytes_per_step"] == want_in
    assert e2e["d2h_bytes_per_step"] == 112

    assert line["gpu_launches"] == 2 * K  # the MX workload's encodes run inside its norm pass
    clk = line["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk) and isinstance(clk["reasons"], list)

    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_threads() and cb["value"] > 0
    assert cb["unit"] == "params/s" and cb["sample"]
    assert cb["single_thread"]["cores"] == 1


def test_bench_default_run_carries_the_other_workloads():
    """The default run also times the 2^24-parameter, GPT-2-small and MXFP8
    workloads in short loops of their own, at full size, with every pass's
    statistics (here on a small headline workload to keep the test short)."""
    line = _line(["--steps", "5", "--warmup", "3", "--workload", "flat65k_p4", "--no-e2e", "--no-cpu-baseline",
                  "--no-alternatives"])
    cfg = line["configs"]
    assert set(cfg) == set(bench.CONFIG_WORKLOADS)
    for name, c in cfg.items():
        wl = synth.workload(name)
        assert c["N"] == wl.n and c["P"] == wl.p and c["value"] > 0 and c["same_batch"]["value"] > 0
        assert c["ms_per_step"] == pytest.approx(wl.n / c["value"] * 1e3, rel=1e-9)
        assert {"norm", "step"} <= set(c["kernels"])
        for k in ("norm", "step"):
            assert c["kernels"][k]["launches"] >= bench.MIN_PASS_SAMPLES and c["kernels"][k]["gbs"] > 0
        assert 0 < c["whole_step_frac"] < 2
        if wl.mx:  # the separate encodes and MX norm pass, timed beside the fused one
            sep = c["separate_encode"]
            assert {"encode", "norm", "step"} <= set(sep["kernels"]) and sep["value"] > 0
