"""bench.py's own arm on the GPU, on small workloads: one JSON line with every
key of the benchmark contract, each holding what it claims (the roofline
fraction is achieved / peak, the e2e byte counts are the bytes the step's
inputs and the scalar block occupy, the launch count is the passes per step
times the timed steps)."""
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
    argv = ["--steps", str(K), "--warmup", str(W), "--workload", workload] + (["--n", str(n)] if n else [])
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

    e2e = line["e2e"]
    assert e2e["unit"] == "params/s" and e2e["value"] > 0 and e2e["serial"] > 0
    # inputs copied every step: the P bf16 buffers, or the P ranks' codes and scales
    want_in = wl.p * total * 2 if not wl.mx else wl.p * (total + total // 32)
    assert e2e["h2d_bytes_per_step"] == want_in
    assert e2e["d2h_bytes_per_step"] == 112

    assert line["gpu_launches"] == (2 + (wl.p if wl.mx else 0)) * K
    clk = line["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk) and isinstance(clk["reasons"], list)

    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_threads() and cb["value"] > 0
    assert cb["unit"] == "params/s" and cb["sample"]
    assert cb["single_thread"]["cores"] == 1
