"""Benchmark: the sharded mixed-precision optimizer step on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload flat3b_p8] [--variant ldg|tma|staged]

A step is one whole optimizer step of the library on one batch of resident
synthetic gradients: the norm pass (reduce-scatter + unscale + global norm +
found-inf + clip decision) and the fused shard step (reduce-scatter +
unscale + clip + AdamW on fp32 w/m/v + bf16 all-gather) over all P
simulated ranks. Default workload: the largest that fits one GPU, N = 3e9
parameters over P = 8 ranks (fp32 w, m, v: 36 GB; bf16 params: 6 GB; two
batches of eight bf16 gradient buffers: 96 GB), gradients N(0, 1e-3) x 1024,
AdamW lr 1e-3, betas 0.9/0.999, eps 1e-8, wd 0.01, clip 1.0. Two gradient
batches (the workload's steps 1 and 2) alternate, so every step reads fresh
gradients; the working set is far larger than the 129 MB L2, so no flush is
needed between steps.

Prints one JSON line (rank 0). ``value`` is parameters updated per second
over the whole job; ``kernels`` gives every pass's mean and spread over at
least 20 launches, each between its own CUDA events, and its bandwidth on
the algorithmic bytes and on the DRAM bytes ncu measured; ``roofline``
describes the fused shard-step pass against the measured HBM bandwidth;
``e2e`` is the same metric through the C ABI with the gradients copied from
page-locked host memory every step and the step scalars read back every step
(step k+1's copy overlapped with step k through two device input slots;
``e2e.serial`` without that overlap); ``configs`` repeats the measurement on
the 2^24-parameter, GPT-2-small and MXFP8 workloads, each in its own short
loop; ``cpu_baseline`` is the oracle timed on the host.

Under torchrun (N > 1) every GPU runs its own independent P-rank problem (no
collective on the data path: the simulated ranks live inside one GPU), so
scaling is weak; the ranks only meet at the barriers around the timed region
and in the max-over-ranks reduction of the time.

``--impl reference`` times the oracle (the plain CPU statement of the same
step) on the host cores instead, on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "optimizer-step params/sec"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
SCALARS_D2H_BYTES = 112  # sizeof the device scalar block zg_get_info copies back
COPY_PIECE = 1 << 30     # bytes per host-to-device copy in the end-to-end leg
ALT_SECONDS = 10.0       # longest timed loop of each alternative variant
E2E_SECONDS = 15.0       # longest timed loop of each end-to-end mode


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU from a
    background thread through NVML (the library nvidia-smi uses), reading
    only. Falls back to polling nvidia-smi when NVML cannot be loaded."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, cuda_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        self._active = False
        self.source = "none"
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            bus = None
            try:
                import torch

                props = torch.cuda.get_device_properties(cuda_index)
                bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            except Exception:
                bus = None
            ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self._nvml, self._handle = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.source = "nvml"
        except OSError:
            self._nvml = None
            self.source = "nvidia-smi"
            self._index = cuda_index

    def _read(self):
        if self._nvml is not None:
            mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz))
            fn = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            fn(self._handle, ctypes.byref(rs))
            return int(mhz.value), int(rs.value)
        out = subprocess.run(
            ["nvidia-smi", f"--id={self._index}", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
             "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10).stdout.strip()
        sm, mx, act = [x.strip() for x in out.split(",")]
        self.max_mhz = int(mx)
        return int(sm), int(act, 16)

    def _loop(self):
        while not self._stop.is_set():
            try:
                s = self._read()
                if self._active:
                    self.samples.append(s)
            except Exception:
                pass
            time.sleep(self.period if self._nvml is not None else 0.2)

    def start(self):
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()

    def region(self, active: bool):
        self._active = active

    def stop(self) -> dict:
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=5)
        mhz = [s for s, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(name for b, name in self.REASONS.items() if bits & b and name != "gpu_idle")
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(mhz), "source": self.source}


# --------------------------------------------------------------------- helpers

def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in d:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """A hash of the CUDA sources with their comments and blank space taken
    out, so that ncu counters stay attached to the code they were taken on
    while a comment is corrected."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "zero_sharded_mixed_flat_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
            text = re.sub(r"//[^\n]*", "", text)                # line comments (no string in these sources holds //)
            h.update(f.encode())
            h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel}/{workload}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("src_hash") != kernel_source_hash():
        return None
    return float(rec["dram_bytes_per_launch"])


def dist_env() -> tuple[int, int, int]:
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------------- oracle leg

def time_oracle(workload, budget_s: float, steps: int, warmup: int = 0) -> dict:
    """Time the oracle's whole step on a contiguous prefix of the flat vector
    (all P ranks). The prefix length is sized so one step takes about
    ``budget_s`` on one host core. Returns params/s and the sample used."""
    import numpy as np

    import oracle
    from zero_sharded_mixed_flat_gb300 import synth

    def run(ns: int, k: int) -> float:
        w0 = synth.init_weights(workload, 0, ns)
        grads = [synth.grads_bf16(workload, 1, r, 0, ns) for r in range(workload.p)]
        opt = oracle.OracleOptimizer(w0)
        t0 = time.perf_counter()
        for _ in range(k):
            if workload.mx:  # each rank encodes its gradient, then the step sums decoded values
                enc = [oracle.mx_encode(g) for g in grads]
                opt.step_mx([c for c, _ in enc], [s for _, s in enc], workload.loss_scale)
            else:
                opt.step(grads, workload.loss_scale)
        return time.perf_counter() - t0

    probe = min(workload.n, 1 << 16)
    rate = probe / max(run(probe, 2) / 2, 1e-9)
    ns = int(min(workload.n, max(4096, rate * budget_s)))
    ns = max(32, ns // 32 * 32)
    if warmup:
        run(ns, warmup)
    el = run(ns, steps)
    return {"value": ns * steps / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {ns} of {workload.n} params, all {workload.p} ranks, {steps} steps, one thread",
            "seconds": el}


def oracle_threaded_steps(workload, ns: int, k: int, ex, threads: int) -> tuple:
    """``k`` oracle steps on the first ``ns`` parameters of the workload, the
    work spread over the executor ``ex`` (``threads`` workers) as contiguous
    index ranges cut at multiples of 32 (the oracle's C calls release the
    interpreter lock):
    reduce-scatter and sum of squares per range (on the MX workload each
    rank's encode per range first), the fp64 partials added in range order,
    one decision, AdamW per range. Same arithmetic as the one-thread oracle;
    the sum of squares differs only by fp64 rounding order. Returns (seconds,
    w, m, v, t, the sums of squares of the steps)."""
    import numpy as np

    import oracle
    from zero_sharded_mixed_flat_gb300 import synth

    hp = oracle.Hparams()
    p = workload.p
    w = synth.init_weights(workload, 0, ns).copy()
    m = np.zeros(ns, np.float32)
    v = np.zeros(ns, np.float32)
    m.fill(0.0)  # touch the pages before the timed region
    v.fill(0.0)
    grads = [synth.grads_bf16(workload, 1, r, 0, ns) for r in range(p)]
    cut = sorted({min(ns, ns * i // threads // 32 * 32) for i in range(threads)} | {ns})
    ranges = [(a, b) for a, b in zip(cut[:-1], cut[1:]) if b > a]
    inv = oracle.inv_scale(workload.loss_scale, p, hp.grad_average)
    t, b1p, b2p = 0, 1.0, 1.0

    def part(ab):
        a, b = ab
        if workload.mx:
            enc = [oracle.mx_encode(g[a:b]) for g in grads]
            g = oracle.mx_reduce_unscale([c for c, _ in enc], [sc for _, sc in enc], 0, b - a, inv)
        else:
            g = oracle.reduce_unscale(grads, a, b, inv)
        return g, oracle.sumsq(g)

    def update(i, dec, res):
        a, b = ranges[i]
        oracle.adamw_range(hp, dec, res[i][0], w[a:b], m[a:b], v[a:b])

    sums = []
    t0 = time.perf_counter()
    for _ in range(k):
        res = list(ex.map(part, ranges))
        total = 0.0
        for _, ss in res:
            total = total + ss
        sums.append(total)
        dec, nxt = oracle.decide(hp, t, b1p, b2p, total)
        if not dec.found_inf:
            list(ex.map(lambda i: update(i, dec, res), range(len(ranges))))
            t, b1p, b2p = nxt
    return time.perf_counter() - t0, w, m, v, t, sums


def time_oracle_threads(workload, budget_s: float, steps: int, threads: int, warmup: int = 0) -> dict:
    """The oracle on ``threads`` host threads (``oracle_threaded_steps``), on
    a prefix sized so one step takes about ``budget_s`` of wall time."""
    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(threads) as ex:
        probe = min(workload.n, 1 << 20)
        rate = probe / max(oracle_threaded_steps(workload, probe, 2, ex, threads)[0] / 2, 1e-9)
        ns = int(min(workload.n, max(1 << 16, rate * budget_s)))
        ns = max(32, ns // 32 * 32)
        if warmup:
            oracle_threaded_steps(workload, ns, warmup, ex, threads)
        el = oracle_threaded_steps(workload, ns, steps, ex, threads)[0]
    return {"value": ns * steps / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {ns} of {workload.n} params, all {workload.p} ranks, {steps} steps, "
                      f"{threads} threads on contiguous ranges", "seconds": el}


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------- bucket overlap

def time_overlap(opt, wl, dev, stream, K: int, gemm_n: int = 8192) -> dict:
    """How much of the optimizer step hides behind a backward pass when the
    norm is taken bucket by bucket as gradients become ready.

    The backward pass is stood in for by one bf16 GEMM (gemm_n^3, cuBLAS) per
    25M-element gradient bucket, all on one stream. Serial: every GEMM, then
    the norm pass, then the step pass. Overlapped: bucket b's norm runs on a
    second stream as soon as GEMM b is done; the step follows the last
    bucket. Reported: times per step and the optimizer time left exposed
    after the backward pass (the part that cannot be hidden)."""
    import torch

    from zero_sharded_mixed_flat_gb300 import synth
    from zero_sharded_mixed_flat_gb300 import binding as zb

    ls = wl.loss_scale
    bks = synth.buckets(wl.n)
    a = torch.randn(gemm_n, gemm_n, device="cuda", dtype=torch.bfloat16)
    b = torch.randn(gemm_n, gemm_n, device="cuda", dtype=torch.bfloat16)
    c = torch.empty(gemm_n, gemm_n, device="cuda", dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in bks]

    def backward():
        for i in range(len(bks)):
            torch.matmul(a, b, out=c)
            done[i].record(stream)

    def serial():
        backward()
        zb.zg_grad_norm(opt.ctx, dev, ls, stream)
        zb.zg_shard_step(opt.ctx, dev, ls, stream)

    def overlapped():
        backward()
        for i, (lo, hi) in enumerate(bks):
            side.wait_event(done[i])
            flags = (zb.ZG_BUCKET_FIRST if i == 0 else 0) | (zb.ZG_BUCKET_LAST if i == len(bks) - 1 else 0)
            zb.zg_grad_norm_bucket(opt.ctx, dev, lo, hi, ls, flags, side)
        zb.zg_shard_step(opt.ctx, dev, ls, side)
        stream.wait_stream(side)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    t_bwd = timed(backward)
    t_serial = timed(serial)
    t_overlap = timed(overlapped)
    info = opt.info(stream)
    assert info.status == 0
    return {"buckets": len(bks), "bucket_elements": bks[0][1] - bks[0][0],
            "backward_stand_in": f"{len(bks)} bf16 GEMMs of {gemm_n}^3 (cuBLAS), one per bucket",
            "backward_ms": t_bwd, "serial_ms": t_serial, "overlapped_ms": t_overlap,
            "optimizer_exposed_serial_ms": t_serial - t_bwd, "optimizer_exposed_overlapped_ms": t_overlap - t_bwd}


# --------------------------------------------------------------------- stage three

def stage3_layers(wl) -> list[tuple[int, int]]:
    """Layer ranges [lo, hi) of the flat vector: for GPT-2 small its
    embeddings, twelve blocks and final norm; otherwise 16 near-equal parts
    cut at multiples of 768."""
    from zero_sharded_mixed_flat_gb300 import synth

    if wl.name == "gpt2small_p8" and wl.n == 124_439_808:
        out, lo, key_prev = [], 0, None
        for name, k in synth.gpt2_small_tensors():
            key = "embed" if name in ("wte", "wpe") else name.split(".")[0]
            if key == key_prev:
                out[-1] = (out[-1][0], lo + k)
            else:
                out.append((lo, lo + k))
            key_prev, lo = key, lo + k
        return out
    cuts = sorted({min(wl.n, round(i * wl.n / 16 / 768) * 768) for i in range(16)} | {wl.n})
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def time_stage3(opt, wl, K: int, peak: float, tokens: int = 8192) -> dict:
    """Stage three's just-in-time parameter gather over a forward sweep.

    Gather alone: every layer's parameters gathered from the P shards, back
    to back (the kernel's bandwidth). Forward stand-in: per layer one bf16
    GEMM of [tokens x 768] by the gathered parameters viewed as [768 x k]
    (2 * tokens flops per parameter, cuBLAS). Serial: gather, then GEMM, layer
    by layer. Overlapped: layer i+1 is gathered on a second stream into the
    other of two buffers while layer i's GEMM runs (that stream at high or at
    equal priority; for bf16 shards also with the copy-engine gather). Each
    sweep is captured once in a CUDA graph and replayed,
    as a per-layer loop runs in production, so host launch costs stay out of
    the GPU times. Reported: per-sweep times and the gather time left exposed."""
    import torch

    from zero_sharded_mixed_flat_gb300 import accounting

    layers = stage3_layers(wl)
    d = 768
    big = max(hi - lo for lo, hi in layers)
    bufs = [torch.empty(big, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    x = torch.randn(tokens, d, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(tokens * (big // d), dtype=torch.bfloat16, device="cuda")
    side_hi = torch.cuda.Stream(priority=-1)  # gather blocks go first whenever GEMM blocks retire
    side_eq = torch.cuda.Stream()
    gathered = [torch.cuda.Event() for _ in layers]
    used = [torch.cuda.Event(), torch.cuda.Event()]

    def gather(i, b, st, dma=False):
        lo, hi = layers[i]
        opt.gather(lo, hi, bufs[b][:hi - lo], st, dma=dma)

    def compute(i, b):
        lo, hi = layers[i]
        k = (hi - lo) // d // 8 * 8  # an aligned leading dimension keeps cuBLAS on its tensor-core kernels
        torch.matmul(x, bufs[b][:k * d].view(d, k), out=y[:tokens * k].view(tokens, k))

    def gathers_only(dma=False):
        def run():
            cur = torch.cuda.current_stream()
            for i in range(len(layers)):
                gather(i, i % 2, cur, dma)
        return run

    def gemms_only():
        for i in range(len(layers)):
            compute(i, i % 2)

    def serial():
        cur = torch.cuda.current_stream()
        for i in range(len(layers)):
            gather(i, i % 2, cur)
            compute(i, i % 2)

    def overlapped(side, dma=False):
        def run():
            cur = torch.cuda.current_stream()
            side.wait_stream(cur)
            gather(0, 0, side, dma)
            gathered[0].record(side)
            for i in range(len(layers)):
                b = i % 2
                if i + 1 < len(layers):
                    if i >= 1:
                        side.wait_event(used[1 - b])  # layer i-1's GEMM is done with that buffer
                    gather(i + 1, 1 - b, side, dma)
                    gathered[i + 1].record(side)
                cur.wait_event(gathered[i])
                compute(i, b)
                used[b].record(cur)
        return run

    def timed(fn):
        fn()  # launch configurations cached before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    mx = getattr(opt, "pcodes", None) is not None
    t_gather = timed(gathers_only())
    t_gemm = timed(gemms_only)
    t_serial = timed(serial)
    t_hi = timed(overlapped(side_hi))
    t_eq = timed(overlapped(side_eq))
    per_param = accounting.mx_gather_bytes_per_param() if mx else accounting.gather_bytes_per_param()
    gbs = per_param * wl.n / (t_gather / 1e3) / 1e9
    flops = 2 * tokens * sum((hi - lo) // d // 8 * 8 * d for lo, hi in layers)
    dma = {}
    if not mx:  # the copy-engine gather (bf16 shards only)
        t_dma = timed(gathers_only(True))
        t_dma_ov = timed(overlapped(side_eq, True))
        dma = {"gather_dma_ms": t_dma, "gather_dma_gbs": per_param * wl.n / (t_dma / 1e3) / 1e9,
               "overlapped_dma_ms": t_dma_ov, "gather_exposed_overlapped_dma_ms": t_dma_ov - t_gemm}
    return {"layers": len(layers), "largest_layer": big, "shards": "MXFP8 codes + scales" if mx else "bf16",
            "timing": "each sweep captured in a CUDA graph, replayed",
            "gather_ms": t_gather, "gather_gbs": gbs, "gather_frac": gbs / peak,
            "gather_bytes_per_param": per_param,
            "forward_stand_in": f"per layer one bf16 GEMM [{tokens} x {d}] x [{d} x layer/{d}] (cuBLAS)",
            "gemm_ms": t_gemm, "gemm_tflops": flops / (t_gemm / 1e3) / 1e12,
            "serial_ms": t_serial, "overlapped_ms": t_hi, "overlapped_equal_priority_ms": t_eq,
            "gather_exposed_serial_ms": t_serial - t_gemm, "gather_exposed_overlapped_ms": t_hi - t_gemm,
            "gather_exposed_overlapped_equal_priority_ms": t_eq - t_gemm,
            **dma,
            "ring_bytes_per_rank_per_sweep": accounting.ring_bytes_sent_per_rank(
                (accounting.MX_BYTES_PER_ELEMENT if mx else accounting.PARAM_BF16) * wl.n, wl.p, "all_gather")}


# --------------------------------------------------------------------- inputs and steps

# The workloads timed beside the headline one, each in its own short loop.
CONFIG_WORKLOADS = ("flat16m_p8", "gpt2small_p8", "mxfp8_128m_p8")
CONFIG_STEPS = {"flat16m_p8": 200, "gpt2small_p8": 40, "mxfp8_128m_p8": 40}
MIN_PASS_SAMPLES = 20


def host_mem_available() -> float:
    """Bytes of host memory the kernel reports as available (inf if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024.0
    except OSError:
        pass
    return float("inf")


class RegisteredHost:
    """A host array page-locked in place with cudaHostRegister, as a torch
    tensor (``t``), in memory the kernel is asked to back with transparent huge
    pages. The GPU reads page-locked host memory through an address
    translation per page: with the Grace host's 64 KB pages a 48 GB source is
    some 750,000 translations and copied at 16-17 GB/s (measured), a 6 GB one
    read eight times at 140-210 GB/s; huge pages cut the translations by four
    orders of magnitude."""

    def __init__(self, shape, np_dtype, torch_dtype):
        import mmap

        import numpy as np
        import torch

        count = int(np.prod(shape))
        nbytes = count * np.dtype(np_dtype).itemsize
        self._map = mmap.mmap(-1, max(nbytes, 1), flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        self.huge = False
        try:
            self._map.madvise(mmap.MADV_HUGEPAGE)
            self.huge = True
        except (AttributeError, OSError, ValueError):
            pass
        self.a = np.frombuffer(self._map, dtype=np_dtype, count=count).reshape(shape)
        self.a.reshape(-1)[:: max(1, 4096 // self.a.itemsize)] = 0  # fault every page in before locking
        rc = int(torch.cuda.cudart().cudaHostRegister(self.a.ctypes.data, self.a.nbytes, 0))
        if rc != 0:
            raise RuntimeError(f"cudaHostRegister of {self.a.nbytes} bytes failed ({rc})")
        self.t = torch.from_numpy(self.a).view(torch_dtype)

    def close(self) -> None:
        """Unlock the pages (the mapping is released with the last reference)."""
        import torch

        if self.a is not None:
            torch.cuda.cudart().cudaHostUnregister(self.a.ctypes.data)
            self.a, self.t = None, None


def load_batches(wl, nbatch: int, keep_host: bool):
    """``nbatch`` gradient batches of the workload (its steps 1, 2, ...), each
    a device tensor [P, P*S] of bf16 whose row r is rank r's buffer, copied to
    the device before anything is timed. With ``keep_host`` batch 0 is drawn
    straight into page-locked host memory (a RegisteredHost), which is
    returned as well (the end-to-end leg copies a step's inputs from it)."""
    import numpy as np
    import torch

    from zero_sharded_mixed_flat_gb300 import synth

    total = synth.padded_len(wl)
    dev, host = [], None
    for b in range(nbatch):
        d = torch.empty((wl.p, total), dtype=torch.bfloat16, device="cuda")
        if b == 0 and keep_host:
            host = RegisteredHost((wl.p, total), np.uint16, torch.int16)
            for r in range(wl.p):
                synth.grads_bf16(wl, b + 1, r, 0, total, out=host.a[r])
            d.view(torch.int16).copy_(host.t)
        else:
            for r in range(wl.p):
                h = synth.grads_bf16(wl, b + 1, r, 0, total)
                d[r].view(torch.int16).copy_(torch.from_numpy(h.view(np.int16)))
        dev.append(d)
    torch.cuda.synchronize()
    return dev, host


class Stepper:
    """Issues whole optimizer steps through the library, cycling over the
    resident gradient batches (a fresh batch every step when there are two).
    On the MX workload a step first encodes the P ranks' gradients (the
    wire payload), then runs the MX norm and step passes."""

    def __init__(self, opt, wl, dev, stream, mx_fused: bool = True):
        import torch

        from zero_sharded_mixed_flat_gb300 import synth

        self.opt, self.wl, self.stream = opt, wl, stream
        self.rows = [list(d.unbind(0)) for d in dev]
        self.k = 0
        self.mx_fused = mx_fused
        if wl.mx:
            total = synth.padded_len(wl)
            self.codes = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(wl.p)]
            self.scales = [torch.empty(total // 32, dtype=torch.uint8, device="cuda") for _ in range(wl.p)]

    def step(self, ev=None, stream=None):
        """One whole step; with events, mark [start, after norm, after step,
        after the encodes] (the last only on the MX workload's separate
        encodes; the fused encode-and-norm pass counts as the norm pass)."""
        from zero_sharded_mixed_flat_gb300 import binding as zb

        st = stream if stream is not None else self.stream
        g = self.rows[self.k % len(self.rows)]
        self.k += 1
        ls = self.wl.loss_scale
        ctx = self.opt.ctx
        if ev is None and not self.wl.mx:
            zb.zg_step(ctx, g, ls, st)
            return
        if ev is not None:
            ev[0].record(st)
        if self.wl.mx and self.mx_fused:
            zb.zg_quant_norm_mxfp8(ctx, g, self.codes, self.scales, ls, st)
        elif self.wl.mx:
            for r in range(self.wl.p):
                zb.zg_quant_mxfp8(g[r], self.codes[r], self.scales[r], self.wl.n, st)
            if ev is not None:
                ev[3].record(st)
            zb.zg_grad_norm_mxfp8(ctx, self.codes, self.scales, ls, st)
        else:
            zb.zg_grad_norm(ctx, g, ls, st)
        if ev is not None:
            ev[1].record(st)
        if self.wl.mx:
            zb.zg_shard_step_mxfp8(ctx, self.codes, self.scales, ls, st)
        else:
            zb.zg_shard_step(ctx, g, ls, st)
        if ev is not None:
            ev[2].record(st)


def time_loop(stepper, K: int, world: int, clocks=None) -> float:
    """Seconds for K back-to-back steps issued as a caller issues them (no
    event between the passes), bracketed by barrier + synchronize and timed
    with CUDA events on the launching stream; the max over ranks."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.region(True)
    e0.record(stepper.stream)
    for _ in range(K):
        stepper.step()
    e1.record(stepper.stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.region(False)
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1) / 1e3, world)


def time_passes(stepper, samples: int) -> dict:
    """Per-pass durations (ms) of ``samples`` steps, each pass bracketed by its
    own events. The events keep the step pass from starting while the norm
    pass drains, so these are the passes' own times, without that overlap."""
    import torch

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(samples)]
    torch.cuda.synchronize()
    for i in range(samples):
        stepper.step(ev[i])
    torch.cuda.synchronize()
    separate = stepper.wl.mx and not stepper.mx_fused
    n0 = 3 if separate else 0
    out = {"norm": [e[n0].elapsed_time(e[1]) for e in ev], "step": [e[1].elapsed_time(e[2]) for e in ev]}
    if separate:
        out["encode"] = [e[0].elapsed_time(e[3]) for e in ev]
    return out


def pass_stats(ms: list[float], bytes_per_launch: float, peak: float, traffic: float | None) -> dict:
    """Mean, median, spread of a pass's launch times, and its bandwidth on the
    algorithmic bytes and (when the ncu counters match the sources) on the
    DRAM bytes ncu measured for the same launch."""
    xs = sorted(ms)
    mean_s = statistics.fmean(xs) / 1e3
    st = {"launches": len(xs), "mean_us": mean_s * 1e6, "median_us": statistics.median(xs) * 1e3,
          "min_us": xs[0] * 1e3, "max_us": xs[-1] * 1e3,
          "stdev_us": statistics.stdev(xs) * 1e3 if len(xs) > 1 else 0.0,
          "algorithmic_bytes": bytes_per_launch, "gbs": bytes_per_launch / mean_s / 1e9,
          "frac": bytes_per_launch / mean_s / 1e9 / peak, "dram_bytes": traffic}
    if traffic:
        st.update(dram_gbs=traffic / mean_s / 1e9, frac_dram=traffic / mean_s / 1e9 / peak)
    return st


def launch_bytes(wl, variant: str, params: str, mx_fused: bool = True) -> tuple[float, float, float]:
    """Algorithmic bytes of one step pass, one norm pass (on the MX workload
    with mx_fused: the pass that also encodes every rank) and the P separate
    encodes."""
    from zero_sharded_mixed_flat_gb300 import accounting

    n, p = wl.n, wl.p
    if wl.mx and mx_fused:
        step = (accounting.staged_shard_step_bytes_per_param() if variant == "staged"
                else accounting.mx_shard_step_bytes_per_param(p))
        norm = (accounting.mx_staged_quant_norm_bytes_per_param(p) if variant == "staged"
                else accounting.mx_quant_norm_bytes_per_param(p))
        return step * n, norm * n, 0.0
    if wl.mx and variant == "staged":
        return (accounting.staged_shard_step_bytes_per_param() * n, accounting.mx_staged_grad_norm_bytes_per_param(p) * n,
                accounting.mx_quant_bytes_per_param() * p * n)
    if wl.mx:
        return (accounting.mx_shard_step_bytes_per_param(p) * n, accounting.mx_grad_norm_bytes_per_param(p) * n,
                accounting.mx_quant_bytes_per_param() * p * n)
    if variant == "staged":
        return accounting.staged_shard_step_bytes_per_param() * n, accounting.staged_grad_norm_bytes_per_param(p) * n, 0.0
    if params == "mxfp8":
        return accounting.mx_params_shard_step_bytes_per_param(p) * n, accounting.grad_norm_bytes_per_param(p) * n, 0.0
    return accounting.shard_step_bytes_per_param(p) * n, accounting.grad_norm_bytes_per_param(p) * n, 0.0


def kernel_names(wl, variant: str, params: str, mx_fused: bool = True) -> tuple[str, str]:
    """Names the ncu counters are recorded under: (step pass, norm pass)."""
    step = ("zg_shard_step_mxfp8" if wl.mx else "zg_shard_step") + \
        {"staged": "_staged", "tma": "" if wl.mx else "_tma"}.get(variant, "")
    if params == "mxfp8":
        step += "_mxparams"
    norm = (("zg_quant_norm_mxfp8" if mx_fused else "zg_grad_norm_mxfp8") if wl.mx else "zg_grad_norm") + \
        ("_staged" if variant == "staged" else "")
    return step, norm


def kernel_block(passes: dict, wl, key: str, variant: str, params: str, peak: float, mx_fused: bool = True) -> dict:
    """Every pass's statistics with its bandwidth (see pass_stats)."""
    b_step, b_norm, b_quant = launch_bytes(wl, variant, params, mx_fused)
    k_step, k_norm = kernel_names(wl, variant, params, mx_fused)
    out = {"step": pass_stats(passes["step"], b_step, peak, recorded_traffic(k_step, key)),
           "norm": pass_stats(passes["norm"], b_norm, peak, recorded_traffic(k_norm, key))}
    if "encode" in passes:
        t = recorded_traffic("zg_quant_mxfp8", key)
        out["encode"] = pass_stats(passes["encode"], b_quant, peak, t * wl.p if t else None)
        out["encode"]["launches_per_sample"] = wl.p
    return out


# --------------------------------------------------------------------- CUDA graphs

def time_graph(stepper, K: int, per_graph: int = 10) -> dict:
    """The same steps captured `per_graph` at a time into one CUDA graph and
    replayed: what launch overhead the eager loop still pays."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        stepper.step(stream=side)  # launch configurations cached before capture
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(per_graph):
            stepper.step(stream=side)
    reps = max(1, K // per_graph)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * per_graph)
    info = stepper.opt.info()
    assert info.status == 0 and not info.found_inf
    return {"value": stepper.wl.n / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps_per_graph": per_graph,
            "steps": reps * per_graph}


# --------------------------------------------------------------------- end to end

def time_e2e(h_in, slot_inputs, step_on, opt, stream, steps: int, world: int) -> dict:
    """Steps fed from pinned host memory, each step's result read back.

    Serial: copy a step's inputs, run the step, read its result, in turn.
    Pipelined (a caller's double buffer): two device slots; step k+1's inputs
    are copied on a second stream while step k runs, and a slot is refilled
    only after the step that read it is done. Both timed regions hold every
    step's copy and every step's result read."""
    import torch

    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(k):
        # pieces of at most COPY_PIECE bytes: one very large host-to-device
        # copy measured well below the link rate on GB300
        for d, h in zip(slot_inputs(k), h_in):
            dflat, hflat = d.reshape(-1), h.reshape(-1)
            step = max(1, COPY_PIECE // hflat.element_size())
            for i in range(0, hflat.numel(), step):
                dflat[i:i + step].copy_(hflat[i:i + step], non_blocking=True)

    def feed(k):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[k])
            copy_in(k)
            copied[k].record(copy_stream)

    def serial(count):
        for _ in range(count):
            copy_in(0)
            step_on(0)
            opt.info(stream)  # device->host read of the step result; synchronises

    def pipelined(count):
        copy_stream.wait_stream(stream)
        feed(0)
        for k in range(count):
            s = k % 2
            stream.wait_event(copied[s])
            step_on(s)
            consumed[s].record(stream)
            if k + 1 < count:
                feed(1 - s)
            opt.info(stream)

    def timed(run):
        run(2)
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(steps)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / 1e3, world) / steps

    s_serial = timed(serial)
    s_pipe = timed(pipelined)
    info = opt.info(stream)
    assert info.status == 0 and not info.found_inf
    return {"s_per_step": s_pipe, "serial_s_per_step": s_serial, "steps": steps,
            "pipeline": "two device input slots; step k+1's inputs copied on a second stream during step k"}


def e2e_leg(stepper, dev, host, max_steps: int, world, step_s: float) -> dict:
    """The same metric through the C ABI with every step's inputs copied
    from pinned host memory and the step scalars read back every step. bf16
    workloads: the P gradient buffers (all P rows in one pinned buffer, copied
    in pieces of at most 1 GiB; where host memory is short, one rank's buffer
    copied into every rank's row). MX workload: the encoded wire payload (codes and
    scales, encoded on the GPU and parked in host memory, as a sending rank
    would transmit them)."""
    import torch

    from zero_sharded_mixed_flat_gb300 import binding as zb

    import numpy as np

    wl, opt, stream, ls = stepper.wl, stepper.opt, stepper.stream, stepper.wl.loss_scale
    p = wl.p
    owned = []  # page-locked buffers made here, unlocked at the end
    if wl.mx:
        for r in range(p):
            zb.zg_quant_mxfp8(dev[0][r], stepper.codes[r], stepper.scales[r], wl.n, stream)
        # rows of the padded length P * S (a multiple of 32): every rank's codes stay 16-byte aligned
        h_in = []
        for bufs in (stepper.codes, stepper.scales):
            h = RegisteredHost((p, bufs[0].numel()), np.uint8, torch.uint8)
            h.t.copy_(torch.stack(bufs).cpu())
            owned.append(h)
            h_in.append(h.t)
        slots = [[torch.empty_like(h, device="cuda") for h in h_in] for _ in range(2)]
        source = "MXFP8 codes + scales of the P ranks (the wire payload), one page-locked buffer each"

        def slot_inputs(k):
            return slots[k]

        def step_on(k):
            c, sc = slots[k]
            zb.zg_step_mxfp8(opt.ctx, list(c.unbind(0)), list(sc.unbind(0)), ls, stream)
    else:
        slots = list(dev) + [torch.empty_like(dev[0]) for _ in range(2 - len(dev))]
        if host is not None:
            h_in = [host.t]
            source = "P bf16 gradient buffers, one page-locked buffer, copied in pieces of at most 1 GiB"

            def slot_inputs(k):
                return [slots[k].view(torch.int16)]
        else:
            row = RegisteredHost((slots[0].shape[1],), np.uint16, torch.int16)
            owned.append(row)
            row.t.copy_(dev[0][0].view(torch.int16))
            h_in = [row.t] * p
            source = ("one rank's pinned bf16 buffer copied into each of the P rank buffers "
                      "(host memory too small for all P)")

            def slot_inputs(k):
                return [slots[k][r].view(torch.int16) for r in range(p)]

        def step_on(k):
            zb.zg_step(opt.ctx, list(slots[k].unbind(0)), ls, stream)

    # each of the two timed loops about E2E_SECONDS long at most, at the
    # host link's rate (K steps when shorter, 200 at most)
    h2d = sum(h.numel() * h.element_size() for h in h_in)
    est = h2d / 150e9 + step_s
    try:
        res = time_e2e(h_in, slot_inputs, step_on, opt, stream,
                       max(3, min(max_steps, 200, int(E2E_SECONDS / est))), world)
    finally:
        torch.cuda.synchronize()
        for h in owned:
            h.close()
    serial = res.pop("serial_s_per_step")
    return {"value": world * wl.n / res.pop("s_per_step"), "unit": UNIT, "serial": world * wl.n / serial, **res,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": SCALARS_D2H_BYTES, "inputs": source,
            # the copies' own rate in the serial loop: the step's bytes over the time not spent in the step
            "h2d_gbs_in_serial_loop": h2d / max(serial - step_s, 1e-9) / 1e9}


# --------------------------------------------------------------------- our arm

def time_variant(name: str, stepper, warmup: int, K: int, samples: int, world: int, peak: float, key: str) -> dict:
    """The same device-resident steps, on the same context and state, with
    another bf16 variant of the library (identical results): whole-step
    params/s and its passes' statistics. The context returns to the default
    variant afterwards."""
    import torch

    from zero_sharded_mixed_flat_gb300 import binding as zb

    opt, wl = stepper.opt, stepper.wl
    if name == "staged":
        if getattr(opt, "stage", None) is None:
            opt.stage = torch.empty(wl.n, dtype=torch.float32, device="cuda")
            zb.zg_bind_grad_stage(opt.ctx, opt.stage)
        zb.zg_set_variant(opt.ctx, zb.ZG_VARIANT_STAGED)
    else:
        zb.zg_set_variant(opt.ctx, {"tma": zb.ZG_VARIANT_TMA, "single": zb.ZG_VARIANT_SINGLE}[name])
    try:
        for _ in range(warmup):
            stepper.step()
        total = time_loop(stepper, K, world)
        # the one-launch step has no passes to time apart: its launches are timed whole
        passes = time_whole_launches(stepper, samples) if name == "single" else time_passes(stepper, samples)
        info = opt.info(stepper.stream)
        assert info.status == 0 and not info.found_inf, info
    finally:
        zb.zg_set_variant(opt.ctx, zb.ZG_VARIANT_LDG)
    b_step, b_norm, _ = launch_bytes(wl, "ldg" if name == "single" else name, "bf16")
    if name == "single":
        t = [recorded_traffic(k, key) for k in kernel_names(wl, "ldg", "bf16")]
        kern = {"whole": pass_stats(passes["whole"], b_step + b_norm, peak, sum(t) if all(t) else None)}
        kern["whole"]["dram_bytes_source"] = "sum of the two-launch passes' ncu DRAM bytes"
    else:
        kern = kernel_block(passes, wl, key, name, "bf16", peak)
    return {"value": world * wl.n * K / total, "unit": UNIT, "ms_per_step": total * 1e3 / K,
            "whole_step_bytes_per_param": (b_step + b_norm) / wl.n,
            "whole_step_frac": (b_step + b_norm) * K / total / 1e9 / peak, "kernels": kern,
            "gpu_launches": (1 if name == "single" else 2) * K}


def time_whole_launches(stepper, samples: int) -> dict:
    """Durations (ms) of ``samples`` whole steps, each between its own events."""
    import torch

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(samples)]
    torch.cuda.synchronize()
    for e in ev:
        e[0].record(stepper.stream)
        stepper.step()
        e[1].record(stepper.stream)
    torch.cuda.synchronize()
    return {"whole": [e[0].elapsed_time(e[1]) for e in ev]}


def bench_config(name: str, warmup: int, samples: int, peak: float, stream, e2e: bool = False) -> dict:
    """One workload in its own short loop: whole steps with a fresh gradient
    batch every step (the workload's steps 1 and 2 alternating), the same
    with one batch repeated (where lines left in L2 by the previous step can
    be read again), and every pass's statistics over ``samples`` launches;
    with ``e2e`` also the end-to-end leg (inputs from host memory)."""
    import torch

    from zero_sharded_mixed_flat_gb300 import binding as zb
    from zero_sharded_mixed_flat_gb300 import synth

    wl = synth.workload(name)
    dev, host = load_batches(wl, 2, keep_host=e2e and not wl.mx)
    opt = zb.ShardedAdamW(wl.n, wl.p, zb.Hparams(), torch.from_numpy(synth.init_weights(wl)))
    st = Stepper(opt, wl, dev, stream)
    for _ in range(warmup):
        st.step()
    K = CONFIG_STEPS[name]
    t_fresh = time_loop(st, K, 1)
    same = Stepper(opt, wl, dev[:1], stream)
    t_same = time_loop(same, K, 1)
    passes = time_passes(st, samples)
    info = opt.info(stream)
    assert info.status == 0 and info.step_t == warmup + 2 * K + samples, info
    b_step, b_norm, b_quant = launch_bytes(wl, "ldg", "bf16")
    whole = b_step + b_norm + b_quant
    kern = kernel_block(passes, wl, name, "ldg", "bf16", peak)
    sum_us = sum(kern[k]["mean_us"] for k in kern)
    out = {"N": wl.n, "P": wl.p, "steps": K, "value": wl.n * K / t_fresh, "unit": UNIT,
           "ms_per_step": t_fresh * 1e3 / K, "whole_step_bytes_per_param": whole / wl.n,
           "whole_step_gbs": whole * K / t_fresh / 1e9, "whole_step_frac": whole * K / t_fresh / 1e9 / peak,
           "grads": "the workload's steps 1 and 2 alternating (a fresh batch every step)",
           "same_batch": {"value": wl.n * K / t_same, "ms_per_step": t_same * 1e3 / K,
                          "whole_step_frac": whole * K / t_same / 1e9 / peak},
           "kernels": kern, "passes_sum_us": sum_us,
           "overlap_us": sum_us - t_fresh * 1e6 / K}
    if wl.mx:
        # the same steps with the P encodes and the MX norm pass (from the
        # stored codes) as separate launches, as a receiving rank runs them
        sep = Stepper(opt, wl, dev, stream, mx_fused=False)
        t_sep = time_loop(sep, K, 1)
        p_sep = time_passes(sep, samples)
        b_s, b_n, b_q = launch_bytes(wl, "ldg", "bf16", mx_fused=False)
        out["separate_encode"] = {
            "value": wl.n * K / t_sep, "ms_per_step": t_sep * 1e3 / K,
            "whole_step_bytes_per_param": (b_s + b_n + b_q) / wl.n,
            "whole_step_frac": (b_s + b_n + b_q) * K / t_sep / 1e9 / peak,
            "kernels": kernel_block(p_sep, wl, name, "ldg", "bf16", peak, mx_fused=False),
            "gpu_launches_per_step": 2 + wl.p}
        info = opt.info(stream)
        assert info.status == 0 and info.step_t == warmup + 3 * K + 2 * samples, info
        del sep
    if e2e:
        out["e2e"] = e2e_leg(st, dev, host, 200, 1, t_fresh / K)
    if host is not None:
        host.close()
    del st, same, opt, dev
    torch.cuda.empty_cache()
    return out


def bench_ours(args, rank: int, world: int, local: int) -> dict | None:
    import torch

    from zero_sharded_mixed_flat_gb300 import synth
    from zero_sharded_mixed_flat_gb300 import binding as zb

    torch.cuda.set_device(local)
    t_setup = time.perf_counter()
    over = {**({"n": args.n} if args.n else {}), **({"p": args.p} if args.p else {})}
    wl = synth.workload(args.workload, **over)
    key = args.workload if not over else f"{args.workload}@{wl.n}" + (f"/P={wl.p}" if args.p else "")
    n, p = wl.n, wl.p
    total = synth.padded_len(wl)
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    samples = max(MIN_PASS_SAMPLES, args.kernel_samples)

    # inputs resident in HBM before timing: two batches of the P gradient
    # buffers (one with --same-grads); with the end-to-end leg, batch 0 is
    # drawn into pinned host memory when the host has room for it
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    host_bytes = p * total * 2
    keep_host = (not args.no_e2e and not wl.mx
                 and host_bytes + 24e9 < host_mem_available() / max(1, local_world))
    dev, host = load_batches(wl, 1 if args.same_grads else 2, keep_host)
    opt = zb.ShardedAdamW(n, p, zb.Hparams(), torch.from_numpy(synth.init_weights(wl)), offload=args.offload)
    if args.params == "mxfp8":
        opt.use_mx_params()
    if args.variant == "staged":
        opt.use_staged()
    else:
        zb.zg_set_variant(opt.ctx, {"tma": zb.ZG_VARIANT_TMA, "single": zb.ZG_VARIANT_SINGLE}.get(
            args.variant, zb.ZG_VARIANT_LDG))
    mx_fused = not args.mx_separate
    stepper = Stepper(opt, wl, dev, stream, mx_fused)
    setup_s = time.perf_counter() - t_setup

    for _ in range(args.warmup):
        stepper.step()
    info = opt.info(stream)
    assert info.status == 0 and not info.found_inf

    K = args.steps
    clocks = ClockSampler(local)
    clocks.start()
    t0 = time.perf_counter()
    t_max = time_loop(stepper, K, world, clocks)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    info = opt.info(stream)
    assert info.status == 0 and info.step_t == args.warmup + K, info
    value = world * n * K / t_max

    # the passes' own times: `samples` more steps, every pass between its own
    # events (the one-launch variant: every whole step between its own events)
    single = args.variant == "single"
    passes = time_whole_launches(stepper, samples) if single else time_passes(stepper, samples)
    info = opt.info(stream)
    assert info.status == 0 and info.step_t == args.warmup + K + samples, info
    b_step, b_norm, b_quant = launch_bytes(wl, "ldg" if single else args.variant, args.params, mx_fused)
    if single:
        kern = {"whole": pass_stats(passes["whole"], b_step + b_norm, peak, None)}
        step_kernel, sk, b_roof = "zg_step (one launch)", kern["whole"], b_step + b_norm
    else:
        kern = kernel_block(passes, wl, key, args.variant, args.params, peak, mx_fused)
        step_kernel, _ = kernel_names(wl, args.variant, args.params, mx_fused)
        sk, b_roof = kern["step"], b_step
    whole_bytes = b_step + b_norm + b_quant
    sum_us = sum(kern[k]["mean_us"] for k in kern)
    kern.update(timing=f"each pass of {samples} further steps between its own CUDA events (no overlap "
                       "between the passes); mean and spread over those launches",
                passes_sum_us=sum_us, whole_step_us=t_max * 1e6 / K, overlap_us=sum_us - t_max * 1e6 / K,
                whole_step_gbs=whole_bytes * K / t_max / 1e9, whole_step_frac=whole_bytes * K / t_max / 1e9 / peak)

    # the other bf16 variants on the same state and inputs, then CUDA graphs
    plain = not wl.mx and args.variant == "ldg" and not args.offload and args.params == "bf16"
    alternatives = {}
    step_s = t_max / K
    if plain and not args.no_alternatives:
        # each variant's timed loop about ALT_SECONDS long at most (K steps when shorter)
        k_alt = max(3, min(K, int(ALT_SECONDS / step_s)))
        for name in ("staged", "tma", "single"):
            alternatives[name] = time_variant(name, stepper, min(args.warmup, k_alt), k_alt, samples, world, peak,
                                              key)
    graph = (time_graph(stepper, max(K, 20)) if plain and not args.no_alternatives and world == 1
             and t_max / K < 2e-3 else None)

    # end to end (refills the resident batches from host memory)
    e2e = None if args.no_e2e else e2e_leg(stepper, dev, host, args.steps, world, step_s)
    if host is not None:
        host.close()

    # copy probe: achievable HBM bandwidth in the same process
    src = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    for _ in range(3):
        zb.zg_probe_copy(src, dst, stream)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(10):
        zb.zg_probe_copy(src, dst, stream)
    c1.record(stream)
    torch.cuda.synchronize()
    kern["probe_copy_gbs"] = 2 * src.numel() * 10 / (c0.elapsed_time(c1) / 1e3) / 1e9
    del src, dst

    overlap = time_overlap(opt, wl, stepper.rows[0], stream, max(3, min(K, 50))) if args.overlap and not wl.mx else None
    stage3 = time_stage3(opt, wl, max(3, min(K, 20)), peak) if args.stage3 else None
    del stepper, opt, dev
    torch.cuda.empty_cache()

    configs = {}
    if world == 1 and not args.no_configs:
        for name in CONFIG_WORKLOADS:
            if name != args.workload:
                configs[name] = bench_config(name, max(args.warmup, 3), samples, peak, stream,
                                             e2e=not args.no_e2e and name != "gpt2small_p8")

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_max * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic: seeded bf16 gradients resident in HBM, "
                + ("one batch (the workload's step 1) every step" if args.same_grads
                   else "the workload's steps 1 and 2 alternating (a fresh batch every step)"),
        "config": {"workload": key, "N": n, "P": p, "loss_scale": wl.loss_scale, "variant": args.variant,
                   "optimizer_state": "pinned host memory (offloaded)" if args.offload else "HBM",
                   "params": args.params,
                   "optimizer": "AdamW lr 1e-3 b 0.9/0.999 eps 1e-8 wd 0.01 clip 1.0",
                   "l2": f"inputs larger than L2: {(total * 2 * p * (1 if args.same_grads else 2) + n * 14) / 1e9:.2f} "
                         "GB working set vs 0.129 GB L2, no flush"},
        "roofline": {"bound": "hbm", "kernel": step_kernel, "achieved": sk["gbs"], "peak": peak,
                     "unit": "GB/s", "frac": sk["gbs"] / peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6800 GB/s",
                     "traffic": sk["dram_bytes"], "frac_dram": sk.get("frac_dram"),
                     "launches_timed": samples, "duration_us": sk["mean_us"], "stdev_us": sk["stdev_us"],
                     "algorithmic_bytes_per_launch": b_roof, "bytes_per_param": b_roof / n},
        "kernels": kern,
        "e2e": e2e,
        "alternatives": alternatives,
        **({"overlap": overlap} if overlap else {}),
        **({"stage3": stage3} if stage3 else {}),
        **({"graph": graph} if graph else {}),
        "configs": configs,
        "gpu_launches": ((1 if single else 2) + (p if wl.mx and not mx_fused else 0)) * K,
        "clocks": clk,
        "setup_s": setup_s,
        "wall_s": wall,
    }
    if args.offload:
        # the fp32 state crosses the host link twice per step (read, then written back)
        out["offload"] = {"state_bytes_over_link_per_step": 24 * n,
                          "link_gbs_in_step_pass": 24 * n / (sk["mean_us"] / 1e6) / 1e9}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on every host thread, and on one
        one = time_oracle(wl, budget_s=2.0, steps=5)
        out["cpu_baseline"] = {**time_oracle_threads(wl, budget_s=0.3, steps=5, threads=host_threads()),
                               "single_thread": {k: one[k] for k in ("value", "unit", "cores", "sample", "seconds")}}
    return out if rank == 0 else None


# --------------------------------------------------------------------- reference arm

def bench_reference(args) -> dict:
    from zero_sharded_mixed_flat_gb300 import synth

    wl = synth.workload(args.workload)
    budget = max(0.01, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    cb = time_oracle_threads(wl, budget_s=budget, steps=args.steps, threads=host_threads(), warmup=args.warmup)
    return {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["seconds"] * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded bf16 gradients)",
        "config": {"workload": args.workload, "N": wl.n, "P": wl.p, "loss_scale": wl.loss_scale,
                   "sample": cb["sample"]},
        "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="flat3b_p8")
    ap.add_argument("--variant", choices=["ldg", "tma", "staged", "single"], default="ldg")
    ap.add_argument("--n", type=int, default=None, help="override the workload's parameter count (small profiling runs)")
    ap.add_argument("--p", type=int, default=None, help="override the workload's rank count (rank-count sweeps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-alternatives", action="store_true", help="skip timing the other bf16 variants")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' short loops (the configs sub-object)")
    ap.add_argument("--same-grads", action="store_true",
                    help="one resident gradient batch every step instead of two alternating")
    ap.add_argument("--kernel-samples", type=int, default=MIN_PASS_SAMPLES,
                    help=f"steps whose passes are timed one by one (at least {MIN_PASS_SAMPLES})")
    ap.add_argument("--params", choices=["bf16", "mxfp8"], default="bf16",
                    help="store the updated parameters as bf16 (default) or MXFP8 codes + scales")
    ap.add_argument("--mx-separate", action="store_true",
                    help="MX workload: the P encodes and the MX norm pass as separate launches")
    ap.add_argument("--overlap", action="store_true",
                    help="also time the bucketed norm overlapped with a stand-in backward pass")
    ap.add_argument("--stage3", action="store_true",
                    help="also time stage three's just-in-time parameter gather over a forward sweep")
    ap.add_argument("--offload", action="store_true",
                    help="fp32 optimizer state in pinned host memory, read and written over the host link")
    args = ap.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    rank, world, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        out = bench_ours(args, rank, world, local)
        if out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
