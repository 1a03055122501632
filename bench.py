"""Throughput of the attention forward on GB300, as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--batch B] [--no-cpu]

A step is one fa_fwd launch over the whole workload (default: B=8, H=32,
N=4096, d=128, causal -- the pages' B = 8, h = 32 example).  The metric is
attention-forward TFLOP/s with 4·B·H·N²·d FLOPs per step, halved under the
causal mask.

* value: inputs resident in HBM; K launches timed with CUDA events on the
  launching stream between two barriers + synchronisations; max over ranks.
  Inputs (Q, K, V: 805 MB at the default workload) are larger than L2, so no
  extra flush is made between launches.
* e2e: the same metric through the public call with host buffers: every step
  copies Q, K, V from pinned host memory to the device, runs fa_fwd and copies
  O and the logsumexp back, all inside the timed region.  As in a serving
  loop, the copies in, the compute and the copies out run on three streams
  with two device buffer sets, so one step's copies overlap its neighbours'
  compute (pipelined_e2e).
* roofline: the attention kernel is tensor-core bound; achieved = algorithmic
  FLOPs per launch / mean launch time, against the measured bf16 GEMM peak
  (frac), the measured sustained peak and NVIDIA's datasheet dense figure;
  beside it the exponential unit's bound (one ex2 per score).
* blocks beside the headline (default run): non_causal (the other half of
  the metric, B=8 H=32 N=4096 d=128), sustained (the headline launch
  repeated for a seconds-long region under the power cap) and one block per
  other configuration, each with its own clocks, launch spread and roofline;
  the small configuration also reports the host cost of a call.
* cpu_baseline: the fp64 CPU oracle timed on the host cores over a bounded
  sample of rows of the same workload (rank 0 only), with all threads and
  with one, and the full tensor's time extrapolated from those rates.
* --impl reference: the oracle alone (the reference arm: the pages ship no
  runnable code), each step a bounded sample of rows.
* --workload ew_*: the fused elementwise chain (bias + GELU + dropout) of
  the pages' fusion discussion; one step is one fa_bias_gelu_dropout launch,
  the metric its algorithmic bytes per second against the HBM copy peak.
* --pass bwd: the backward instead (fa_bwd: gradients dQ, dK, dV for a given
  dO, d = 64 or 128); a step is one fa_bwd call (three launches: prepare, main,
  dQ conversion) and the FLOPs are those of its five matrix products,
  10·B·H·N²·d, halved under the causal mask.

With N > 1 (torchrun) every rank runs its own copy of the workload on its own
GPU: the (batch, head) problems are independent, so there is no data-path
collective ("scaling": "weak"); only the timing barrier and the max-over-ranks
reduction communicate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16) and % of GB300 dense BF16 peak, causal & non-causal"
BWD_METRIC = "attention bwd TFLOP/s (bf16) and % of GB300 dense BF16 peak"
DECODE_METRIC = "attention decode (split-KV): KV-cache bytes read per second"
EW_METRIC = "fused bias+GELU+dropout (bf16): HBM bytes per second (x, bias, keep mask read once, y written once)"

FWD_SOURCES = ("fa_fwd_kernel.cuh", "ptx.cuh", "fa_api.cu")
BWD_SOURCES = ("fa_bwd_kernel.cuh", "fa_fwd_kernel.cuh", "ptx.cuh", "fa_api.cu")
EW_SOURCES = ("fa_ew_kernel.cuh", "ptx.cuh", "fa_api.cu")
# DRAM bytes (read + write) per launch from one ncu capture, keyed by workload
# name and pass, with the sha256 of the kernel sources it was taken on;
# reported as roofline.traffic only while the sources still hash the same.
# The captures ran B = 2 of the same workload (a smaller launch that still
# exceeds L2) and are scaled by 4 to a full launch: every (batch, head)
# problem moves the same bytes.  profiles/ holds the summaries and commands.
MEASURED_TRAFFIC = {
    ("b8_h32_n4096_d128_causal", "fwd"): {
        "sources": FWD_SOURCES,
        "sha256": "71c822ee1441c996e8c74e94626390f0491be3ee090d4363e3ec00823ce04fa0",
        "bytes": 4 * (201_403_136 + 45_192_448),
        "captured_on": "B=2, H=32, N=4096, d=128, causal; x4"},
    ("b8_h32_n4096_d128_causal", "bwd"): {
        "sources": BWD_SOURCES,
        "sha256": "ebffbaadb9cb155cd97c994938d0223b429299257acebd694938e8c3c24ce022",
        "bytes": 4 * (406_204_672 + 218_182_656),
        "captured_on": "B=2, H=32, N=4096, d=128, causal; main kernel only; x4"},
    ("ew_b8_t4096_d4096_p0.1", "ew"): {
        "sources": EW_SOURCES,
        "sha256": "a1280852145bf2c19457b9232e3cdebf52f538b2b2dcaad13f9d284a96159670",
        "bytes": 285_297_664 + 210_903_040,
        "captured_on": "the full workload (537 MB on the device)"},
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's published dense BF16 tensor figure for one GB300 GPU: its HGX B300
# table gives 36 PFLOPS of FP16/BF16 for 8 GPUs with 2:4 sparsity, i.e. 4.5
# sparse and 2.25 dense PFLOPS per GPU.  A second denominator beside the
# measured cuBLAS peak.
DATASHEET_BF16_TFLOPS = 2250.0
DATASHEET_SOURCE = ("NVIDIA HGX B300 specification (nvidia.com/en-us/data-center/hgx/): 36 PFLOPS FP16/BF16 "
                    "for 8 GPUs, with sparsity; dense per GPU = 36 / 8 / 2")
# The special-function unit's exponential: one ex2.approx.f32 warp
# instruction issues every 4.2 cycles per SM sub-partition (a probe of
# back-to-back independent ex2 on this GPU), i.e. 4 x 32 / 4.2 = 30.5
# exponentials per cycle per SM.  The kernel evaluates one per score.
EX2_CYCLES_PER_WARP_INSTR = 4.2


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling captures)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline time budget")
    ap.add_argument("--no-blocks", action="store_true",
                    help="headline only: skip the non-causal, sustained and per-configuration blocks")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of the sustained block's timed region")
    return ap.parse_args(argv)


def kernel_sources_sha256(names=FWD_SOURCES) -> str:
    import hashlib

    hsh = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "io_aware_attention_gb300", "csrc", name), "rb") as f:
            hsh.update(f.read())
    return hsh.hexdigest()


def measured_traffic(workload_name: str, pass_: str = "fwd"):
    rec = MEASURED_TRAFFIC.get((workload_name, pass_))
    if rec is None or rec["sha256"] != kernel_sources_sha256(rec["sources"]):
        return None
    return rec["bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank value over the default process group; the value itself
    when no group is initialised.  The reduction tensor lives on `device` (the
    rank's GPU under NCCL, the CPU under gloo)."""
    import torch
    import torch.distributed as distm

    if not (distm.is_available() and distm.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    distm.all_reduce(t, op=distm.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs its own copy of the workload (weak
    scaling), timed by the slowest rank."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def pipelined_e2e(n_steps, host_in, out_like, compute, nbuf=2, lanes=1):
    """Milliseconds per step of n_steps end-to-end steps.  A step copies the
    pinned host tensors `host_in` to the device, runs `compute(ins, outs,
    stream)` (the public call, writing the device tensors `outs`) and copies
    `outs` back to pinned host tensors.  nbuf sets of device buffers; the
    copies in, the compute and the copies out run on separate streams linked
    by events, so that the next step's copies in and the previous step's
    copies out run while a step computes, as a serving loop would.  With
    lanes > 1 each direction's copies are cut into pieces spread over that
    many streams (measured slower for the attention steps: one stream per
    direction is the default).  Every copy of every step
    lies inside the timed region (CUDA events from before the first copy in
    to after the last copy out)."""
    import torch

    dev_in = [[torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in host_in] for _ in range(nbuf)]
    dev_out = [[torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in out_like] for _ in range(nbuf)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in out_like] for _ in range(nbuf)]
    s_in = [torch.cuda.Stream() for _ in range(lanes)]
    s_out = [torch.cuda.Stream() for _ in range(lanes)]
    s_comp = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(lanes)] for _ in range(nbuf)]
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [[torch.cuda.Event() for _ in range(lanes)] for _ in range(nbuf)]

    def pieces(dsts, srcs):
        # (dst, src) views of about equal size, `lanes` per tensor
        out = []
        for d, h in zip(dsts, srcs):
            dv, hv = d.view(-1), h.view(-1)
            n = dv.numel()
            step = -(-n // lanes)
            out += [(dv[i:i + step], hv[i:i + step]) for i in range(0, n, step)]
        return out

    plan_in = [pieces(dev_in[b], host_in) for b in range(nbuf)]
    plan_out = [pieces(host_out[b], dev_out[b]) for b in range(nbuf)]

    def run(n):
        for i in range(n):
            b = i % nbuf
            for j, s in enumerate(s_in):
                if i >= nbuf:
                    s.wait_event(ev_comp[b])  # the step that last used buffer set b has read its inputs
                with torch.cuda.stream(s):
                    for d, h in plan_in[b][j::lanes]:
                        d.copy_(h, non_blocking=True)
                ev_in[b][j].record(s)
                s_comp.wait_event(ev_in[b][j])
            if i >= nbuf:
                for e in ev_out[b]:
                    s_comp.wait_event(e)  # ... and its outputs have been copied out
            compute(dev_in[b], dev_out[b], s_comp)
            ev_comp[b].record(s_comp)
            for j, s in enumerate(s_out):
                s.wait_event(ev_comp[b])
                with torch.cuda.stream(s):
                    for h, d in plan_out[b][j::lanes]:
                        h.copy_(d, non_blocking=True)
                ev_out[b][j].record(s)

    run(nbuf + 1)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    start.record(s_comp)
    for s in s_in:
        s.wait_event(start)
    run(n_steps)
    end = torch.cuda.Event(enable_timing=True)
    for e in ev_out[(n_steps - 1) % nbuf]:
        s_comp.wait_event(e)
    for b in range(nbuf):
        for e in ev_out[b]:
            s_comp.wait_event(e)
    end.record(s_comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / n_steps


E2E_OVERLAP = "copies in / compute / copies out on three streams, two device buffer sets"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


def timed_region(step, n, stream, gpu_index, barrier, label):
    """Milliseconds of n calls of step() on `stream` (CUDA events), between a
    barrier and a synchronisation on both sides, with nvidia-smi clock
    samples taken while they run (gpu_index None: no sampling) and an NVTX
    range around the launches."""
    import torch

    sampler = ClockSampler(gpu_index) if gpu_index is not None else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push(label)
    ev0.record(stream)
    for _ in range(n):
        step()
    ev1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    return ev0.elapsed_time(ev1), clocks


def single_launch_stats(step, stream, n=30):
    """Median, standard deviation and minimum of n single launches, each
    bracketed by its own events."""
    import torch

    pairs = []
    for _ in range(n):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in pairs]
    return {"n": len(ms), "median_ms": round(statistics.median(ms), 5), "stdev_ms": round(statistics.stdev(ms), 5),
            "min_ms": round(min(ms), 5)}


def mufu_bound(w, ms_per_step: float, sm_mhz, sms: int):
    """Time bound of the exponentials: one ex2 per score the method computes
    (B*H*N^2, half of it under the causal mask), at the special-function
    unit's measured rate and the median SM clock of the timed region."""
    if not sm_mhz:
        return None
    scores = w.B * w.H * w.N * w.N * (0.5 if w.causal else 1.0)
    rate = sms * 4 * 32 / EX2_CYCLES_PER_WARP_INSTR * sm_mhz * 1e6
    bound_ms = scores / rate * 1e3
    return {"ex2_per_s": round(rate / 1e12, 3), "unit": "Tex2/s", "scores_per_launch": scores,
            "bound_ms": round(bound_ms, 5), "frac": round(bound_ms / ms_per_step, 4), "sm_mhz": sm_mhz,
            "rate": f"{sms} SMs x 4 x 32 / {EX2_CYCLES_PER_WARP_INSTR} ex2 per cycle at the median SM clock"}


def tensor_roofline(w, flops: float, ms_per_step: float, peaks, peak_src, clocks, sms: int, kernel: str):
    """The forward's roofline entry: algorithmic FLOPs per launch over the
    launch time, against the measured bf16 burst peak (the denominator of
    frac), the sustained peak and the datasheet figure; and the exponential
    unit's bound, with the tighter of the two bounds named."""
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    tensor_ms = flops / (peak * 1e12) * 1e3
    mufu = mufu_bound(w, ms_per_step, clocks.get("sm_mhz") if clocks else None, sms)
    executed = executed_flops(w)
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_source": f"bf16_tflops (burst), {peak_src}",
            "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", peak)), 4),
            "frac_of_datasheet": round(achieved / DATASHEET_BF16_TFLOPS, 4),
            "datasheet_tflops": DATASHEET_BF16_TFLOPS, "kernel": kernel, "alg_flops_per_launch": flops,
            "executed_flops_per_launch": executed, "executed_over_algorithmic": round(executed / flops, 4),
            "executed_frac": round(executed / (ms_per_step * 1e-3) / 1e12 / peak, 4),
            "tensor_bound_ms": round(tensor_ms, 5), "mufu": mufu}
    if mufu:
        roof["binding"] = "tensor" if tensor_ms >= mufu["bound_ms"] else "mufu"
        roof["frac_of_binding"] = round(max(tensor_ms, mufu["bound_ms"]) / ms_per_step, 4)
    return roof


def executed_flops(w) -> float:
    """The tensor work the forward kernel executes per launch, beside the
    algorithmic 4·B·H·N²·d (halved when causal): whole 128 × 128 tiles
    (the causal diagonal ones and a ragged tail included) at the kernel's
    head size D (64 or 128; smaller d are zero-padded), and the P·V product
    at N = D + 16 (the ones block that makes l~).  Per tile 2·128²·D for S
    and 2·128²·(D + 16) for P·V; per head M² tiles, or M(M + 1)/2 under the
    causal mask, M = ceil(N / 128)."""
    D = 64 if w.d <= 64 else 128
    M = (w.N + 127) // 128
    tiles = M * (M + 1) // 2 if w.causal else M * M
    return float(w.B * w.H * tiles * 2 * 128 * 128 * (2 * D + 16))


def fwd_kernel_name(w) -> str:
    D = 64 if w.d <= 64 else 128
    return f"fa::fa_fwd_kernel<{D},{str(w.causal).lower()},{str(w.d != D).lower()},*>"


def fwd_block(fa, w, dev, stream, peaks, peak_src, sms, rank, barrier, min_seconds=0.25, min_steps=20,
              host_cost=False):
    """One workload of the default run, beside the headline: its own inputs,
    timed region (at least min_seconds and min_steps launches), clocks, launch
    spread and roofline."""
    import torch

    from io_aware_attention_gb300 import iomodel
    from io_aware_attention_gb300.workloads import make_qkv

    flops = iomodel.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    q, k, v = (t.to(dev) for t in make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

    def step():
        fa.fwd_into(q, k, v, o, lse, w.causal, w.scale)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    probe_ms, _ = timed_region(step, 5, stream, None, lambda: None, "probe")
    n = max(min_steps, int(min_seconds / max(probe_ms / 5 * 1e-3, 1e-7)) + 1)
    ms, clocks = timed_region(step, n, stream, torch.cuda.current_device() if rank == 0 else None, barrier,
                              f"fa_fwd {w.name}")
    if fa.check_device_status() != 0:
        raise RuntimeError(f"kernel reported a timed-out wait ({w.name})")
    ms_per_step = max_over_ranks(ms, dev) / n
    blk = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
           "steps": n, "ms_per_step": round(ms_per_step, 5), "value": round(flops / (ms_per_step * 1e-3) / 1e12, 2),
           "unit": "TFLOP/s", "timed_s": round(ms / 1e3, 3),
           "roofline": tensor_roofline(w, flops, ms_per_step, peaks, peak_src, clocks, sms, fwd_kernel_name(w)),
           "launch_stats": single_launch_stats(step, stream), "clocks": clocks}
    if host_cost:
        blk["host_us_per_call"] = host_call_cost(fa, q, k, v, o, lse, w, stream)
    del q, k, v, o, lse
    return blk


def host_call_cost(fa, q, k, v, o, lse, w, stream, n=200):
    """Host microseconds per call, launches not waited for: the raw C-ABI call
    (ctypes, arguments prepared once) and the Python binding (shape, dtype
    and device checks, then the same call)."""
    import ctypes

    import torch

    lib = fa.library()
    vp = ctypes.c_void_p
    args = (vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()), vp(lse.data_ptr()),
            w.B, w.H, w.N, w.d, int(w.causal), float(w.scale), vp(stream.cuda_stream))
    out = {}
    for name, call in (("c_abi", lambda: lib.fa_fwd(*args)),
                       ("binding", lambda: fa.fwd_into(q, k, v, o, lse, w.causal, w.scale))):
        call()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            call()
        dt = time.perf_counter() - t0
        torch.cuda.synchronize()
        out[name] = round(dt / n * 1e6, 2)
    return out


def cpu_oracle_rate(w, q, k, v, budget_s: float, seed: int = 7):
    """Times the fp64 oracle on a bounded sample of rows; returns a dict with
    TFLOP/s, the threads used and a description of the sample."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(seed)

    def flops_of(rows):
        vis = (rows + 1) if w.causal else np.full_like(rows, w.N)
        return float(np.sum(4.0 * w.d * vis))

    def run(n, threads=0):
        bh = rng.integers(0, w.B * w.H, size=n, dtype=np.int64)
        row = rng.integers(0, w.N, size=n, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.causal, w.scale, bh, row, threads=threads)
        return time.perf_counter() - t0, flops_of(row)

    threads = oracle.max_threads()
    n = 32
    dt, fl = run(n)
    while dt < 0.5 and n < (1 << 20):  # calibrate
        n *= 4
        dt, fl = run(n)
    rate = fl / dt
    total_n = n
    total_t = dt
    total_f = fl
    main_budget = 0.8 * budget_s
    n_big = max(n, int(n * (main_budget - total_t) / max(dt, 1e-9)))
    if total_t < main_budget:
        dt, fl = run(n_big)
        total_n, total_t, total_f = n_big, dt, fl
        rate = fl / dt
    # One thread, on a sample sized to the rest of the budget.
    per_row_one_thread = total_t / total_n * threads  # assumes near-linear thread scaling
    n1 = max(8, int(0.2 * budget_s / max(per_row_one_thread, 1e-9)))
    dt1, fl1 = run(n1, threads=1)
    rate1 = fl1 / dt1
    full = iomodel_flops(w)
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{total_n} random (b,h,row) rows of the same workload, fp64, "
                      f"{total_t:.1f} s; FLOPs = 4*d*visible keys per row",
            "single_thread": {"value": rate1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"{n1} random rows, {dt1:.1f} s"},
            "extrapolated_full_tensor_s": {"all_threads": round(full / rate, 1), "one_thread": round(full / rate1, 1),
                                           "how": "extrapolated: the workload's FLOPs / the sampled rate"}}


def iomodel_flops(w) -> float:
    from io_aware_attention_gb300 import iomodel

    return iomodel.attention_flops(w.B, w.H, w.N, w.d, w.causal)


def decode_bytes(w) -> int:
    """Algorithmic bytes of one decode step: K and V read once, q read, O and
    the logsumexp written."""
    return 2 * w.B * w.H * w.Nk * w.d * 2 + 2 * w.B * w.H * w.Nq * w.d * 2 + w.B * w.H * w.Nq * 4


def decode_oracle_rate(w, q, k, v, budget_s: float, seed: int = 7):
    """The fp64 oracle on a bounded random sample of query rows of the same
    decode workload; bytes of K and V per row processed per second."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(seed)
    row_bytes = 2 * w.Nk * w.d * 2

    def run(n):
        bh = rng.integers(0, w.B * w.H, size=n, dtype=np.int64)
        row = rng.integers(0, w.Nq, size=n, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.attention_rect_rows(q, k, v, w.causal, w.scale, bh, row)
        return time.perf_counter() - t0

    n = 4
    dt = run(n)
    while dt < min(0.5, budget_s / 4) and n < (1 << 16):  # calibrate
        n *= 2
        dt = run(n)
    if dt < budget_s / 2:  # then one sample sized to the budget
        n = max(n, int(n * budget_s / max(dt, 1e-9)))
        dt = run(n)
    return n, dt, n * row_bytes / dt / 1e9


def run_decode(args, w, rank, world, local):
    """One step = one fa_decode call over the whole (B, H, Nk) cache."""
    import torch
    import torch.distributed as distm

    import io_aware_attention_gb300 as fa
    from io_aware_attention_gb300.workloads import make_decode_qkv

    nbytes = decode_bytes(w)
    config = {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
              "scale": "1/sqrt(d)", "inputs": "Q,K,V iid N(0,1) bf16, seeded", "per_gpu_problem": True,
              "parallelism": f"replicas x{args.gpus}",
              "l2": f"K,V {2 * w.B * w.H * w.Nk * w.d * 2 / 1e6:.0f} MB > 129 MB L2 (no flush)"}
    q_h, k_h, v_h = make_decode_qkv(w)
    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        steps, warm = args.steps, max(args.warmup, 3)
        for _ in range(warm):
            decode_oracle_rate(w, q_h, k_h, v_h, 0.2)
        tot_b, tot_t, n_rows = 0.0, 0.0, 0
        for _ in range(steps):
            n, dt, _ = decode_oracle_rate(w, q_h, k_h, v_h, 0.5)
            tot_b += n * 2 * w.Nk * w.d * 2
            tot_t += dt
            n_rows = n
        value = tot_b / tot_t / 1e9
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": steps, "warmup": warm, "ms_per_step": 1e3 * tot_t / steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                                 "sample": f"{n_rows} random (b,h,row) query rows per step, fp64 two-pass oracle; "
                                           "bytes = K and V of the rows' heads"},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return 0

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        distm.init_process_group("nccl", device_id=dev)
        pg = True
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    ws_bytes = fa.decode_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, w.causal)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 2 if ws_bytes else 1

    for _ in range(max(args.warmup, 3)):
        fa.decode_into(q, k, v, o, lse, ws, w.causal, w.scale)
    torch.cuda.synchronize()
    if fa.check_device_status() != 0:
        raise RuntimeError("decode reported an error during warm-up")
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if pg:
        distm.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        fa.decode_into(q, k, v, o, lse, ws, w.causal, w.scale)
    ev1.record(stream)
    torch.cuda.synchronize()
    if pg:
        distm.barrier()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_per_step = ms / args.steps
    value = nbytes * world / (ms_per_step * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in (q_h, k_h, v_h)]
        n_e2e = max(3, min(args.steps, 5))

        # The workspace is shared: every compute runs on the one compute stream.
        def decode_step(ins, outs, s):
            fa.decode_into(*ins, *outs, ws, w.causal, w.scale, stream=s)

        ems = max_over_ranks(pipelined_e2e(n_e2e, host_in, (o, lse), decode_step), dev)
        e2e = {"value": nbytes * world / (ems * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ems,
               "steps": n_e2e, "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (q, k, v)),
               "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * lse.element_size(),
               "overlap": E2E_OVERLAP}

    peaks, peak_src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = nbytes / (ms_per_step * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"hbm_gbs (copy), {peak_src}",
            "kernel": f"fa::dec::fa_decode_partial_kernel<{w.d},*> + combine", "traffic": None,
            "alg_bytes_per_launch": nbytes}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        n, dt, rate = decode_oracle_rate(w, q_h, k_h, v_h, args.cpu_seconds)
        cpu = {"value": rate, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"{n} random (b,h,row) query rows, fp64, {dt:.1f} s; bytes = K and V of each row's head"}
    if rank == 0:
        line = {"metric": DECODE_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if pg:
        distm.destroy_process_group()
    return 0


def bwd_flops(w) -> float:
    """FLOPs of one backward: five N x N x d products per (batch, head)
    (S = QK^T recomputed, dP = dO V^T, dV = P^T dO, dK = dS^T Q, dQ = dS K),
    2 flops per multiply-add, halved under the causal mask."""
    f = 10.0 * w.B * w.H * w.N * w.N * w.d
    return f / 2 if w.causal else f


def bwd_oracle_rate(w, q, k, v, do, budget_s: float, max_heads: int = 64):
    """The fp64 oracle backward on whole heads of the workload (a head is the
    smallest unit: its gradients need every row), as many as fit the budget.
    Returns (heads, seconds, TFLOP/s) with the FLOPs of bwd_flops per head."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(11)
    flat = lambda t: t.reshape(w.B * w.H, 1, 1, w.N, w.d)
    per_head = 10.0 * w.N * w.N * w.d * (0.5 if w.causal else 1.0)
    heads, total = 0, 0.0
    while heads < max_heads and (heads == 0 or total < budget_s):
        bh = int(rng.integers(0, w.B * w.H))
        ins = [flat(t)[bh].contiguous() for t in (q, k, v, do)]
        t0 = time.perf_counter()
        oracle.attention_bwd(*ins, w.causal, w.scale)
        total += time.perf_counter() - t0
        heads += 1
    return heads, total, heads * per_head / total / 1e12


def run_bwd(args, w, config, rank, world, local):
    """One step = one fa_bwd call (prepare, main kernel, dQ conversion) over the
    whole workload, with O and the logsumexp from fa_fwd computed once."""
    import torch
    import torch.distributed as distm

    import io_aware_attention_gb300 as fa
    from io_aware_attention_gb300.workloads import make_qkv, make_random_qkv

    flops = bwd_flops(w)
    config = dict(config, **{"pass": "bwd", "dO": "iid N(0,1) bf16, seeded (seed + 500)"})
    config["l2"] = (f"inputs {6 * w.B * w.H * w.N * w.d * 2 / 1e6:.0f} MB (q, k, v, o, dO + dq/dk/dv outputs) "
                    "> 129 MB L2 (no flush)")
    q_h, k_h, v_h = make_qkv(w)
    do_h = make_random_qkv(w.B, w.H, w.N, w.d, w.seed + 500)[0]
    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        warm = max(args.warmup, 3)
        steps = args.steps
        bwd_oracle_rate(w, q_h, k_h, v_h, do_h, 0.0, max_heads=1)  # first call: page in, build
        heads, dt, rate = bwd_oracle_rate(w, q_h, k_h, v_h, do_h, budget_s=60.0, max_heads=max(1, steps))
        line = {"impl": "reference", "metric": BWD_METRIC, "value": rate, "unit": "TFLOP/s", "n_gpus": world,
                "steps": heads, "warmup": 1, "ms_per_step": 1e3 * dt / heads, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
                                 "sample": f"{heads} whole random (b,h) heads, one per step (a head is the "
                                           "oracle backward's smallest unit), fp64, at most 60 s"},
                "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return 0

    if w.d not in (64, 128):
        raise SystemExit(f"the backward kernel takes d = 64 or 128; workload {w.name} has d = {w.d}")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        distm.init_process_group("nccl", device_id=dev)
        pg = True
    q, k, v, do = q_h.to(dev), k_h.to(dev), v_h.to(dev), do_h.to(dev)
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.bwd_into(q, k, v, o, lse, do, dq, dk, dv, ws, w.causal, w.scale)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if fa.check_device_status() != 0:
        raise RuntimeError("backward reported a timed-out wait during warm-up")
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if pg:
        distm.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if pg:
        distm.barrier()
    clocks = sampler.stop() if sampler else None
    if fa.check_device_status() != 0:
        raise RuntimeError("backward reported a timed-out wait in the timed region")
    ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_per_step = ms / args.steps
    value = job_tflops(flops, world, ms_per_step)

    e2e = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in (q_h, k_h, v_h)] + [o.cpu().pin_memory(), lse.cpu().pin_memory(),
                                                              do_h.pin_memory()]
        n_e2e = max(3, min(args.steps, 10))

        # The workspace is shared: every compute runs on the one compute stream.
        def bwd_step(ins, outs, s):
            fa.bwd_into(*ins, *outs, ws, w.causal, w.scale, stream=s)

        ems = max_over_ranks(pipelined_e2e(n_e2e, host_in, (dq, dk, dv), bwd_step), dev)
        tb = q.numel() * q.element_size()
        e2e = {"value": job_tflops(flops, world, ems), "unit": "TFLOP/s", "ms_per_step": ems,
               "steps": n_e2e, "h2d_bytes_per_step": 5 * tb + lse.numel() * 4, "d2h_bytes_per_step": 3 * tb,
               "overlap": E2E_OVERLAP}

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_source": f"bf16_tflops (burst), {peak_src}",
            "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", peak)), 4),
            "frac_of_datasheet": round(achieved / DATASHEET_BF16_TFLOPS, 4),
            "kernel": f"fa::bwd::fa_bwd_kernel<{w.d},{str(w.causal).lower()}>; the timed launch is the whole "
                      "fa_bwd call (prepare + main + dQ conversion), so this is a lower bound for the main kernel",
            "traffic": measured_traffic(w.name, "bwd"), "alg_flops_per_launch": flops,
            "traffic_kernel": "main kernel only (fa_bwd_kernel), DRAM read + write per launch"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        heads, dt, rate = bwd_oracle_rate(w, q_h, k_h, v_h, do_h, args.cpu_seconds)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"{heads} whole random (b,h) heads of the workload, fp64 backward, {dt:.1f} s"}
    if rank == 0:
        line = {"metric": BWD_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": 3 * args.steps, "clocks": clocks, "pct_of_peak": round(100 * achieved / peak, 2)}
        print(json.dumps(line), flush=True)
    if pg:
        distm.destroy_process_group()
    return 0


def ew_bytes(w) -> int:
    """Algorithmic bytes of one fused step: x read and y written once (bf16),
    the packed keep mask and the bias read once."""
    n = w.rows * w.cols
    return 4 * n + ((n + 31) // 32) * 4 + 2 * w.cols


def ew_oracle_rate(w, x, b, keep, budget_s: float):
    """The fp64 oracle on the first rows of the workload, as many as fit the
    budget; algorithmic bytes of those rows per second."""
    import numpy as np

    import oracle

    words = keep.numpy().view(np.uint32)
    rows = 64
    while True:
        t0 = time.perf_counter()
        oracle.bias_gelu_dropout(x[:rows], b, words, w.p)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or rows >= w.rows:
            break
        rows = min(w.rows, rows * 4)
    n = rows * w.cols
    return rows, dt, (4 * n + n / 8 + 2 * w.cols) / dt / 1e9


def run_ew(args, w, rank, world, local):
    """One step = one fa_bias_gelu_dropout launch over the whole tensor."""
    import torch
    import torch.distributed as distm

    import io_aware_attention_gb300 as fa
    from io_aware_attention_gb300.workloads import make_ew_inputs

    nbytes = ew_bytes(w)
    config = {"workload": w.name, "rows": w.rows, "cols": w.cols, "p": w.p,
              "inputs": "x ~ N(0,4) bf16, bias ~ N(0,1) bf16, keep bits Bernoulli(1-p), seeded",
              "per_gpu_problem": True, "parallelism": f"replicas x{args.gpus}",
              "l2": f"x + y {4 * w.rows * w.cols / 1e6:.0f} MB > 129 MB L2 (no flush)"}
    x_h, b_h, k_h = make_ew_inputs(w.rows, w.cols, w.p, w.seed)
    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        ew_oracle_rate(w, x_h, b_h, k_h, 0.5)
        tot_b, tot_t, rows = 0.0, 0.0, 0
        for _ in range(min(args.steps, 20)):
            rows, dt, rate = ew_oracle_rate(w, x_h, b_h, k_h, 2.0)
            tot_b += rate * dt * 1e9
            tot_t += dt
        value = tot_b / tot_t / 1e9
        steps = min(args.steps, 20)
        line = {"impl": "reference", "metric": EW_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": steps, "warmup": 1, "ms_per_step": 1e3 * tot_t / steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                                 "sample": f"the first {rows} rows per step, fp64"},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return 0

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        distm.init_process_group("nccl", device_id=dev)
        pg = True
    x, b, keep = x_h.to(dev), b_h.to(dev), k_h.to(dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.bias_gelu_dropout(x, b, keep, w.p, out=y)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if pg:
        distm.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if pg:
        distm.barrier()
    clocks = sampler.stop() if sampler else None
    ms_per_step = max_over_ranks(ev0.elapsed_time(ev1), dev) / args.steps
    value = nbytes * world / (ms_per_step * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        host_in = [x_h.pin_memory(), b_h.pin_memory(), k_h.pin_memory()]
        n_e2e = max(3, min(args.steps, 10))

        def ew_step(ins, outs, s):
            fa.bias_gelu_dropout(ins[0], ins[1], ins[2], w.p, out=outs[0], stream=s)

        ems = max_over_ranks(pipelined_e2e(n_e2e, host_in, (y,), ew_step), dev)
        e2e = {"value": nbytes * world / (ems * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ems, "steps": n_e2e,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (x, b, keep)),
               "d2h_bytes_per_step": y.numel() * y.element_size(), "overlap": E2E_OVERLAP}

    peaks, peak_src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = nbytes / (ms_per_step * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"hbm_gbs (copy), {peak_src}",
            "kernel": "fa::ew::fa_bias_gelu_dropout_kernel<false>", "traffic": measured_traffic(w.name, "ew"),
            "alg_bytes_per_launch": nbytes}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        rows, dt, rate = ew_oracle_rate(w, x_h, b_h, k_h, args.cpu_seconds)
        cpu = {"value": rate, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"the first {rows} rows of the workload, fp64, {dt:.1f} s"}
    if rank == 0:
        line = {"metric": EW_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if pg:
        distm.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    from io_aware_attention_gb300 import iomodel
    from io_aware_attention_gb300.workloads import DECODE_WORKLOADS, EW_WORKLOADS, HEADLINE, WORKLOADS, Workload

    if args.workload in EW_WORKLOADS:
        return run_ew(args, EW_WORKLOADS[args.workload], rank, world, local)

    if args.workload in DECODE_WORKLOADS:
        wd = DECODE_WORKLOADS[args.workload]
        if args.batch:
            from io_aware_attention_gb300.workloads import DecodeWorkload
            wd = DecodeWorkload(wd.name + f"_b{args.batch}", args.batch, wd.H, wd.Nq, wd.Nk, wd.d, wd.causal, wd.seed,
                                wd.sample_rows)
        return run_decode(args, wd, rank, world, local)
    wname = args.workload or HEADLINE
    w = WORKLOADS[wname]
    if args.batch:
        w = Workload(w.name + f"_b{args.batch}", args.batch, w.H, w.N, w.d, w.causal, w.seed,
                     w.q_mult, w.spike_every, w.spike_mult, w.sample_rows)
    flops = iomodel.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    inputs = "Q,K,V iid N(0,1) bf16, seeded"
    if w.q_mult != 1.0 or w.spike_every:
        inputs += f"; Q x{w.q_mult:g}; every {w.spike_every}th key row x{w.spike_mult:g}"
    in_mb = 3 * w.B * w.H * w.N * w.d * 2 / 1e6
    config = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
              "scale": "1/sqrt(d)", "inputs": inputs,
              "per_gpu_problem": True, "parallelism": f"replicas x{args.gpus}",
              "l2": (f"inputs {in_mb:.0f} MB > 129 MB L2 (no flush)" if in_mb > 129 else
                     f"inputs {in_mb:.1f} MB fit in L2 (not flushed: warm-cache figure)")}

    if args.pass_ == "bwd":
        return run_bwd(args, w, config, rank, world, local)
    if args.impl == "reference":
        return run_reference(args, w, flops, config, rank, world)

    import torch
    import torch.distributed as distm

    import io_aware_attention_gb300 as fa
    from io_aware_attention_gb300.workloads import make_qkv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        distm.init_process_group("nccl", device_id=dev)
        pg = True

    def barrier():
        if pg:
            distm.barrier()

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks, peak_src = load_peaks()
    q_h, k_h, v_h = make_qkv(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fwd_into(q, k, v, o, lse, w.causal, w.scale)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if fa.check_device_status() != 0:
        raise RuntimeError("kernel reported a timed-out wait during warm-up")

    # ---- the headline: exactly args.steps launches
    ms, clocks = timed_region(step, args.steps, stream, torch.cuda.current_device() if rank == 0 else None,
                              barrier, f"fa_fwd {w.name} x{args.steps}")
    if fa.check_device_status() != 0:
        raise RuntimeError("kernel reported a timed-out wait in the timed region")
    ms = max_over_ranks(ms, dev)
    ms_per_step = ms / args.steps
    launch_stats = single_launch_stats(step, stream)
    value = job_tflops(flops, world, ms_per_step)

    # ---- end to end through the public call with host buffers
    e2e = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in (q_h, k_h, v_h)]

        def fwd_step(ins, outs, s):
            fa.fwd_into(*ins, *outs, w.causal, w.scale, stream=s)

        n_e2e = max(3, min(args.steps, 20))
        barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("fa_fwd end to end")
        ems = max_over_ranks(pipelined_e2e(n_e2e, host_in, (o, lse), fwd_step), dev)
        torch.cuda.nvtx.range_pop()
        barrier()
        h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
        d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
        e2e = {"value": job_tflops(flops, world, ems), "unit": "TFLOP/s",
               "ms_per_step": ems, "steps": n_e2e, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "overlap": E2E_OVERLAP}

    roof = tensor_roofline(w, flops, ms_per_step, peaks, peak_src, clocks, sms, fwd_kernel_name(w))
    roof["traffic"] = measured_traffic(w.name)
    roof["alg_bytes_per_launch"] = iomodel.attention_min_bytes(w.B, w.H, w.N, w.d)

    # ---- beside the headline (default run only): the other half of the
    # metric (non-causal), the same launch over a seconds-long region (the
    # power-capped figure), and the other configurations.
    blocks = {}
    if not args.no_blocks and args.workload is None and not args.batch:
        # sustained: the headline launch repeated for args.sustained_seconds
        n_sus = max(args.steps, int(args.sustained_seconds / (launch_stats["median_ms"] * 1e-3)) + 1)
        sus_ms, sclocks = timed_region(step, n_sus, stream, torch.cuda.current_device() if rank == 0 else None,
                                     barrier, f"fa_fwd {w.name} sustained x{n_sus}")
        if fa.check_device_status() != 0:
            raise RuntimeError("kernel reported a timed-out wait in the sustained region")
        sus_per = max_over_ranks(sus_ms, dev) / n_sus
        sroof = tensor_roofline(w, flops, sus_per, peaks, peak_src, sclocks, sms, fwd_kernel_name(w))
        if sclocks and sclocks.get("sm_mhz"):
            # time x clock: launch time at the maximum SM clock, if the work
            # scaled with the clock
            sroof["ms_per_step_at_max_clock"] = round(sus_per * sclocks["sm_mhz"] / sclocks["sm_max_mhz"], 5)
        blocks["sustained"] = {"workload": w.name, "steps": n_sus, "timed_s": round(sus_ms / 1e3, 3),
                               "ms_per_step": round(sus_per, 5),
                               "value": round(flops / (sus_per * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                               "roofline": sroof, "clocks": sclocks}
        del q, k, v, o, lse
        torch.cuda.empty_cache()
        others = [("non_causal", "b8_h32_n4096_d128", {}),
                  ("config_b1_h2_n256_d64", "b1_h2_n256_d64", {"host_cost": True, "min_steps": 200}),
                  ("config_b4_h16_n2048_d128_causal", "b4_h16_n2048_d128_causal", {}),
                  ("config_b1_h32_n32768_d128_causal", "b1_h32_n32768_d128_causal", {}),
                  ("config_b16_h16_n8192_d64_spiky", "b16_h16_n8192_d64_spiky", {})]
        for key, name, kw in others:
            blocks[key] = fwd_block(fa, WORKLOADS[name], dev, stream, peaks, peak_src, sms, rank, barrier, **kw)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_oracle_rate(w, q_h, k_h, v_h, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3),
                "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps, "clocks": clocks, "launch_stats": launch_stats,
                "pct_of_peak": round(100 * roof["frac"], 2), "datasheet": DATASHEET_SOURCE}
        line.update(blocks)
        print(json.dumps(line), flush=True)
    if pg:
        distm.destroy_process_group()
    return 0


def run_reference(args, w, flops_full, config, rank, world):
    """The reference arm: the fp64 CPU oracle, timed on the host cores, each
    step a bounded random sample of rows of the same workload."""
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from io_aware_attention_gb300.workloads import make_qkv

    q, k, v = make_qkv(w)
    rng = np.random.default_rng(99)
    steps, warm = args.steps, max(args.warmup, 3)
    per_step_budget = min(0.25, 90.0 / max(1, steps + warm))

    def sample(n):
        return (rng.integers(0, w.B * w.H, size=n, dtype=np.int64),
                rng.integers(0, w.N, size=n, dtype=np.int64))

    def step(n):
        bh, row = sample(n)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.causal, w.scale, bh, row)
        dt = time.perf_counter() - t0
        vis = (row + 1) if w.causal else np.full_like(row, w.N)
        return dt, float(np.sum(4.0 * w.d * vis))

    n = 8
    dt, _ = step(n)
    while dt < per_step_budget / 4 and n < (1 << 18):
        n *= 2
        dt, _ = step(n)
    n = max(1, int(n * per_step_budget / max(dt, 1e-9)))
    for _ in range(warm):
        step(n)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(steps):
        dt, fl = step(n)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": 1e3 * tot_t / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{n} random (b,h,row) rows per step, fp64 two-pass "
                                       "oracle; FLOPs = 4*d*visible keys per row"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
