#!/usr/bin/env python3
"""Benchmark of the fa_fwd attention forward on GB300.

One step = one forward pass (one fa_fwd launch) over the whole workload, with
the inputs resident in HBM. Prints ONE JSON line (rank 0):

  value         whole-job TFLOP/s (4*B*H*M*N*D per head pass, x1/2 when
                causal), device-timed with CUDA events over exactly --steps
                steps, barrier + synchronize on both sides, max over ranks.
  e2e           the same metric through the public call with host buffers:
                each step copies Q, K, V from pinned host memory, runs the
                forward, and copies O and LSE back. For the bf16 forward this
                is fa_fwd_host, which overlaps the copies with the kernel in
                chunks of heads; otherwise plain copies around the call.
  roofline      the kernel's achieved TFLOP/s (per-launch CUDA events) against
                the measured dense-BF16 peak.
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample of the same
                workload on this host's cores (rank 0 only).
  clocks        SM clocks and throttle reasons sampled during the timed region.

``--impl reference`` times the oracle instead (the reference arm): each step
is a bounded sample of the workload on the host cores.

Multi-GPU (torchrun): every rank runs its own full replica of the workload
(the work units are independent; there is no data exchange), so scaling is
weak and ``value`` is the sum over ranks of the work divided by the slowest
rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd attention TFLOP/s (4·B·H·M·N·D, causal ×½), % of BF16 tensor-core peak"
METRIC_BWD = "bwd attention TFLOP/s (10·B·H·M·N·D: five M·N·D products, causal ×½)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "causal_b8_h32_s4096_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 1 s of work)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU seconds for the oracle sample")
    ap.add_argument("--splitkv", type=int, default=None, metavar="S",
                    help="time fa_fwd_splitkv with S key-range splits (0 = the library's suggestion)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size B (smaller cases for profiler captures)")
    ap.add_argument("--seq", type=int, default=None,
                    help="override the workload's sequence lengths M = N (studies of unit length)")
    ap.add_argument("--noncausal", action="store_true", help="run the workload without the causal mask")
    ap.add_argument("--f32-path", choices=["ieee", "x3"], default="ieee",
                    help="fp32 workloads: exact CUDA-core fa_fwd_f32 (ieee) or tensor-core fa_fwd_f32x3 (x3)")
    ap.add_argument("--warm", action="store_true",
                    help="do not flush L2 between timed steps even when a step's inputs fit in it")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward pass fa_bwd on the workload")
    ap.add_argument("--per-config", choices=["auto", "on", "off"], default="auto",
                    help="also time the other benchmark workloads after the headline one (auto: on for the "
                         "default forward workload on one GPU)")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi in the background during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="fa_clocks_", suffix=".csv")
            self._f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self._f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        return summarize_clocks(rows)


# Sources of each path's kernels; a recorded ncu traffic figure is reported
# only while these hash to the value it was taken with.
KERNEL_SOURCES = ["fa_bf16_kernel.cuh", "fa_bf16_q1.cuh", "ptx.cuh", "fa_internal.h", "fa_api.cu",
                  "fa_bf16_d64.cu", "fa_bf16_d96.cu", "fa_bf16_d128.cu"]
X3_SOURCES = ["fa_f32x3.cu", "ptx.cuh", "fa_internal.h", "fa_api.cu"]
PROFILES = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles")
TRAFFIC_FILE = os.path.join(PROFILES, "fa_fwd_bf16_dram_traffic.json")
X3_TRAFFIC_FILE = os.path.join(PROFILES, "fa_fwd_f32x3_dram_traffic.json")


def kernel_sources_sha(sources=None) -> str:
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "flashattention_fa_fwd_gb300", "csrc")
    for name in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(workload: str, path: str = "bf16"):
    """DRAM bytes (read + written) of one step of a path on this workload
    (bf16: the one kernel launch; x3: the split pre-pass plus the attention
    kernel), from the ncu capture recorded under profiles/, or None when
    there is none or the kernel sources changed since it was taken."""
    file, sources = (X3_TRAFFIC_FILE, X3_SOURCES) if path == "x3" else (TRAFFIC_FILE, KERNEL_SOURCES)
    try:
        with open(file) as f:
            rec = json.load(f)
        if rec.get("kernel_sha") != kernel_sources_sha(sources):
            return None
        e = rec["workloads"].get(workload)
        return None if e is None else int(e["dram_bytes_read"]) + int(e["dram_bytes_write"])
    except (OSError, ValueError, KeyError):
        return None


def summarize_clocks(rows):
    """Median SM clock, max clock and the throttle reasons seen (any sample)."""
    def num(x):
        try:
            return float(x)
        except ValueError:
            return None

    sm = [num(r[1]) for r in rows if num(r[1]) is not None]
    mx = [num(r[2]) for r in rows if num(r[2]) is not None]
    reasons = set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for r in rows:
        for name, val in zip(names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(rows),
            "power_w_max": max((num(r[3]) for r in rows if num(r[3]) is not None), default=None)}


def clocks_rejected(clk) -> bool:
    if any(r in BAD_REASONS for r in clk.get("reasons", [])):
        return True
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.5 * mx and not clk.get("reasons"))


# --------------------------------------------------------- multi-rank glue

def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def whole_job_value(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """TFLOP/s over all ranks: every rank does flops_per_step per step."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w, target_s: float):
    """Times the fp64 oracle on sampled query rows of workload w's heads.

    Returns (TFLOP/s under the metric's convention, seconds, rows, cores,
    description). Heads are added (256 sampled rows each, all rows when M is
    smaller) until the sample has taken about target_s seconds.
    """
    import numpy as np

    from flashattention_fa_fwd_gb300.inputs import head_tensor, sample_rows
    from oracle import attention_rows

    flops = 0.0
    secs = 0.0
    nrows = 0
    heads = 0
    for bh in range(w.B * w.H):
        qh = head_tensor(w.wid, 0, bh, w.M, w.D, w.sigma_qk, w.dtype)
        kh = head_tensor(w.wid, 1, bh, w.N, w.D, w.sigma_qk, w.dtype)
        vh = head_tensor(w.wid, 2, bh, w.N, w.D, w.sigma_v, w.dtype)
        rows = sample_rows(w.wid, bh, w.M, 256)
        t0 = time.perf_counter()
        attention_rows(qh, kh, vh, w.scale, w.causal, rows)
        secs += time.perf_counter() - t0
        vis = np.minimum(rows + 1, w.N) if w.causal else np.full(rows.size, w.N)
        flops += 4.0 * w.D * float(vis.sum())
        nrows += int(rows.size)
        heads += 1
        if secs >= target_s:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"{nrows} sampled query rows over {heads} heads of {w.name} ({w.N} keys each, fp64 numpy oracle, "
            f"{secs:.1f} s)")
    return flops / secs / 1e12, secs, nrows, int(cores), desc


def oracle_step_fn(w, rows_per_step: int):
    """One reference-arm step: the oracle on a fixed sample of rows."""
    import numpy as np

    from flashattention_fa_fwd_gb300.inputs import head_tensor, sample_rows
    from oracle import attention_rows

    qh = head_tensor(w.wid, 0, 0, w.M, w.D, w.sigma_qk, w.dtype)
    kh = head_tensor(w.wid, 1, 0, w.N, w.D, w.sigma_qk, w.dtype)
    vh = head_tensor(w.wid, 2, 0, w.N, w.D, w.sigma_v, w.dtype)
    rows = sample_rows(w.wid, 0, w.M, rows_per_step)
    vis = np.minimum(rows + 1, w.N) if w.causal else np.full(rows.size, w.N)
    flops = 4.0 * w.D * float(vis.sum())

    def step():
        attention_rows(qh, kh, vh, w.scale, w.causal, rows)

    return step, flops, int(rows.size)


def reference_arm(args, w, rank, world):
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    steps = args.steps if args.steps is not None else 10
    rows_per_step = min(w.M, 256)
    step, flops, nrows = oracle_step_fn(w, rows_per_step)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    value = flops * steps / dt / 1e12
    sample = f"each step: {nrows} sampled query rows of head 0 of {w.name} (fp64 numpy oracle)"
    model, blas = host_cpu()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), sample=sample),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": model, "blas": blas},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm

# Dense bf16 tensor-core FLOPs per clock per SM: NVIDIA's published dense
# BF16 figure for Blackwell (2.25 PFLOP/s per GPU) at its boost clock, which
# is also what one tcgen05 128x128x16 MMA every 64 cycles delivers
# (2 * 128 * 128 * 16 / 64). TF32 runs at half that rate.
BF16_FLOP_PER_CLK_SM = 8192
TF32_FLOP_PER_CLK_SM = 4096

# Workloads timed after the headline one, in the same run (per_config).
PER_CONFIG = ["f32_single_head_m256_n512_d64", "gpt2m_b64_h16_s1024_d64", "causal_b8_h32_s4096_d128",
              "cross_b2_h8_m1000_n3000_d96_peaked", "long_causal_b1_h8_s65536_d64"]


def spec_peak(sms: int, mhz: float, per_clk: int, what: str):
    """SMs x SM clock x per-SM dense rate, in TFLOP/s, with its derivation."""
    return sms * mhz * 1e6 * per_clk / 1e12, f"{sms} SMs x {mhz:.0f} MHz x {per_clk} dense {what} FLOP/clk/SM"


def host_cpu():
    """The host's CPU model and numpy's BLAS, for the CPU baseline."""
    import platform

    import numpy as np

    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        model = platform.processor() or platform.machine()
    blas = "unknown"
    try:
        b = np.__config__.CONFIG["Build Dependencies"]["blas"]
        blas = f"{b.get('name')} {b.get('version')}"
    except (AttributeError, KeyError, TypeError):
        pass
    return f"{model} ({platform.machine()})", blas


def time_steps(step, steps, stream, dev, flush=None, local_rank=0, world=1):
    """Runs exactly `steps` calls of step() between a barrier + synchronize
    on each side, each bracketed by CUDA events on `stream` (after an L2
    flush on the same stream when `flush` is given), with nvidia-smi
    sampling the clocks. Returns (per-launch ms, total ms of the steps,
    clocks)."""
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_begin.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total = sum(per_launch) if flush is not None else t_begin.elapsed_time(t_end)  # flushes are not the workload
    return per_launch, total, clocks


def launch_stats(per_launch):
    return {"mean": statistics.mean(per_launch), "median": statistics.median(per_launch), "min": min(per_launch),
            "n": len(per_launch)}


def l2_note(flush, step_in_bytes):
    if flush is None and step_in_bytes > 129e6:
        return f"inputs larger than L2 ({step_in_bytes / 2**20:.0f} MiB read per step vs 129 MB L2)"
    if flush is not None:
        return (f"L2 flushed before every timed step (256 MiB written; inputs {step_in_bytes / 2**20:.1f} MiB); "
                "value from the steps' own CUDA events")
    return "inputs fit in L2 (warm, --warm)"


def calibrate(step, stream, dev, target_ms, lo, hi):
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(5):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    per = e0.elapsed_time(e1) / 5
    return int(min(hi, max(lo, math.ceil(target_ms / max(per, 1e-3)))))


def per_config_line(fa, name, dev, stream, peaks, sms, local_rank, splitkv=False, warm=False, cpu_baseline=False):
    """One other workload of the benchmark, timed in the same run: at least
    50 steps (about 0.4 s of device time), median and min per-launch time,
    roofline against both denominators, clocks."""
    import torch

    from flashattention_fa_fwd_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    bf16 = w.dtype == "bf16"
    tdtype = torch.bfloat16 if bf16 else torch.float32
    host = make_inputs(w)
    q, k, v = (torch.from_numpy(x).to(dev).to(tdtype) for x in host)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.M, dtype=torch.float32, device=dev)
    api, splits = ("fa_fwd" if bf16 else "fa_fwd_f32"), 1
    if splitkv:
        splits = fa.fa_fwd_splitkv_suggest(w.B, w.H, w.M, w.N, w.causal)
        ws = torch.empty(max(fa.fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.M, w.D, splits), 16), dtype=torch.uint8,
                         device=dev)
        api = f"fa_fwd_splitkv ({splits} splits, the library's suggestion)"

        def step():
            fa.fa_fwd_splitkv(q, k, v, o, lse, w.scale, w.causal, num_splits=splits, workspace=ws)
    elif bf16:
        def step():
            fa.fa_fwd(q, k, v, o, lse, w.scale, w.causal)
    else:
        def step():
            fa.fa_fwd_f32(q, k, v, o, lse, w.scale, w.causal)
    for _ in range(3):
        step()
    if fa.fa_get_device_status() != fa.FA_OK:
        raise SystemExit(f"device status after the warm-up of {name}")
    steps = calibrate(step, stream, dev, 400.0, 50, 5000)
    step_in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flush = torch.empty(64 * 2**20, dtype=torch.float32, device=dev) if step_in_bytes <= 129e6 and not warm else None
    per_launch, total, clocks = time_steps(step, steps, stream, dev, flush, local_rank)
    if fa.fa_get_device_status() != fa.FA_OK:
        raise SystemExit(f"device status after timing {name}")
    ls = launch_stats(per_launch)
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    if bf16:
        peak, bound = float(peaks["bf16_tflops"]), "tensor"
        pspec, pspec_src = spec_peak(sms, mhz, BF16_FLOP_PER_CLK_SM, "bf16")
    else:
        peak, bound = sms * 128 * 2 * mhz * 1e6 / 1e12, "alu"
        pspec, pspec_src = peak, f"derived: {sms} SMs x 128 fp32 lanes x 2 FLOP x {mhz:.0f} MHz (fp32 FMA)"
    achieved = w.flops / (ls["mean"] * 1e-3) / 1e12
    l2 = l2_note(flush, step_in_bytes)
    del q, k, v, o, lse, flush
    torch.cuda.empty_cache()
    cpu = oracle_config_timing(w, host) if cpu_baseline else None
    del host
    return {
        "value": w.flops * steps / (total * 1e-3) / 1e12, "unit": UNIT, "steps": steps, "api": api,
        "dtype": w.dtype, "config": dict(w.describe(), kv_splits=splits, l2=l2),
        "launch_ms": ls,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                     "achieved_median": w.flops / (ls["median"] * 1e-3) / 1e12,
                     "peak_spec": pspec, "peak_spec_source": pspec_src, "frac_of_spec": achieved / pspec,
                     "traffic": recorded_traffic(name) if bf16 and splits == 1 else None},
        "clocks": clocks, "clocks_rejected": clocks_rejected(clocks),
        "cpu_baseline": cpu,
    }


# Workloads whose oracle the per-config CPU baseline runs in full; the others
# are timed on sampled query rows (the 64K-token workload: 256 rows of each
# of its 8 heads, as its parity test) and extrapolated to the whole workload.
CPU_FULL = ("f32_single_head_m256_n512_d64", "gpt2m_b64_h16_s1024_d64", "cross_b2_h8_m1000_n3000_d96_peaked")


def oracle_config_timing(w, host):
    """The fp64 oracle on this host's cores for workload w (inputs as the GPU
    got them): in full where that takes seconds, else on sampled rows."""
    import numpy as np

    from flashattention_fa_fwd_gb300.inputs import sample_rows
    from oracle import attention, attention_rows

    q, k, v = host
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model, blas = host_cpu()
    out = {"unit": UNIT, "cores": int(cores), "kind": "oracle", "cpu_model": model, "blas": blas}
    if w.name in CPU_FULL:
        t0 = time.perf_counter()
        attention(q, k, v, w.scale, w.causal)
        secs = time.perf_counter() - t0
        out.update(value=w.flops / secs / 1e12, seconds=secs, sample=f"the whole workload ({w.name}, fp64 numpy oracle)")
        return out
    qf, kf, vf = (x.reshape(w.B * w.H, x.shape[-2], w.D) for x in (q, k, v))
    flops, secs, nrows = 0.0, 0.0, 0
    for bh in range(w.B * w.H):
        rows = sample_rows(w.wid, bh, w.M, 256)
        t0 = time.perf_counter()
        attention_rows(qf[bh], kf[bh], vf[bh], w.scale, w.causal, rows)
        secs += time.perf_counter() - t0
        vis = np.minimum(rows + 1, w.N) if w.causal else np.full(rows.size, w.N)
        flops += 4.0 * w.D * float(vis.sum())
        nrows += int(rows.size)
    out.update(value=flops / secs / 1e12, seconds=secs,
               sample=f"{nrows} sampled query rows of {w.name} (256 per head, fp64 numpy oracle)",
               extrapolated_full_seconds=secs * w.flops / flops)
    return out


def gpu_arm(args, w, rank, world, local_rank):
    import numpy as np
    import torch

    import flashattention_fa_fwd_gb300 as fa
    from flashattention_fa_fwd_gb300.inputs import make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the fa_fwd arm")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    fa.load_library()
    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    bf16 = w.dtype == "bf16"
    tdtype = torch.bfloat16 if bf16 else torch.float32
    q_np, k_np, v_np = make_inputs(w)
    hq, hk, hv = (torch.from_numpy(x).to(tdtype).pin_memory() for x in (q_np, k_np, v_np))
    del q_np, k_np, v_np
    q, k, v = (t.to(dev) for t in (hq, hk, hv))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.M, dtype=torch.float32, device=dev)
    call = fa.fa_fwd if bf16 else fa.fa_fwd_f32
    splits = 1
    if args.splitkv is not None and bf16:
        splits = args.splitkv or fa.fa_fwd_splitkv_suggest(w.B, w.H, w.M, w.N, w.causal)
        ws = torch.empty(max(fa.fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.M, w.D, splits), 16),
                         dtype=torch.uint8, device=dev)

        def call(q_, k_, v_, o_, l_, scale_, causal_):
            fa.fa_fwd_splitkv(q_, k_, v_, o_, l_, scale_, causal_, num_splits=splits, workspace=ws)
    x3 = not bf16 and args.f32_path == "x3"
    if x3:
        ws_x3 = torch.empty(max(fa.fa_fwd_f32x3_workspace_bytes(w.B, w.H, w.N, w.D), 16), dtype=torch.uint8,
                            device=dev)

        def call(q_, k_, v_, o_, l_, scale_, causal_):
            fa.fa_fwd_f32x3(q_, k_, v_, o_, l_, scale_, causal_, workspace=ws_x3)
    stream = torch.cuda.current_stream(dev)

    def step():
        call(q, k, v, o, lse, w.scale, w.causal)

    bwd = args.pass_ == "bwd"
    flops = w.flops
    if bwd:
        if not bf16 or splits > 1:
            raise SystemExit("--pass bwd times fa_bwd: a bf16 workload, without --splitkv")
        call(q, k, v, o, lse, w.scale, w.causal)        # the forward whose O and LSE the backward reads
        gen = torch.Generator(device=dev).manual_seed(7)
        dout = torch.randn(q.shape, device=dev, generator=gen).to(torch.bfloat16)
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        ws_bwd = torch.empty(max(fa.fa_bwd_workspace_bytes(w.B, w.H, w.M), 16), dtype=torch.uint8, device=dev)
        flops = w.flops * 2.5    # five products instead of the forward's two

        def step():
            fa.fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, w.scale, w.causal, workspace=ws_bwd)

    for _ in range(max(args.warmup, 3)):
        step()
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise SystemExit(f"device status after warm-up: {fa.fa_status_string(st)}")

    # Default step count: about one second of device time, at least 50 steps.
    if args.steps is None:
        steps = calibrate(step, stream, dev, 1000.0, 50, 5000)
        steps = int(max_over_ranks(float(steps), world, dev))
    else:
        steps = args.steps

    # A step whose inputs fit in L2 (129 MB) would find them there: unless --warm, write 256 MiB
    # on the same stream before every timed step, and take the time from the steps' own events.
    step_in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    if bwd:
        step_in_bytes += sum(t.numel() * t.element_size() for t in (o, lse, dout))
    flush = None
    if step_in_bytes <= 129e6 and not args.warm:
        flush = torch.empty(64 * 2**20, dtype=torch.float32, device=dev)
    l2 = l2_note(flush, step_in_bytes)
    per_launch, timed_ms, clocks = time_steps(step, steps, stream, dev, flush, local_rank, world)
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise SystemExit(f"device status after the timed region: {fa.fa_status_string(st)}")
    max_ms = max_over_ranks(timed_ms, world, dev)
    value = whole_job_value(flops, steps, world, max_ms)
    ls = launch_stats(per_launch)
    achieved = flops / (ls["mean"] * 1e-3) / 1e12
    del flush

    # End to end through the public call with host buffers.
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    e2e_api = "host copies + device call"
    if bwd:
        hdo = dout.cpu().pin_memory()
        ho.copy_(o)
        hl.copy_(lse)
        hdq, hdk, hdv = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ho, hl, hdo))
        d2h = sum(t.numel() * t.element_size() for t in (hdq, hdk, hdv))

        def e2e_step():
            for dst, src in ((q, hq), (k, hk), (v, hv), (o, ho), (lse, hl), (dout, hdo)):
                dst.copy_(src, non_blocking=True)
            fa.fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, w.scale, w.causal, workspace=ws_bwd)
            for dst, src in ((hdq, dq), (hdk, dk), (hdv, dv)):
                dst.copy_(src, non_blocking=True)
    elif bf16 and splits == 1:
        e2e_api = "fa_fwd_host (copies overlapped with the kernel, default chunks)"
        ws_host = torch.empty(max(fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.M, w.N, w.D, 0), 256),
                              dtype=torch.uint8, device=dev)
        del q, k, v, o, lse   # the pipelined call stages through its own workspace
        torch.cuda.empty_cache()

        def e2e_step():
            fa.fa_fwd_host(hq, hk, hv, ho, hl, w.scale, w.causal, workspace=ws_host, device=dev,
                           stream=stream)
    else:
        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            call(q, k, v, o, lse, w.scale, w.causal)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize(dev)
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(x0.elapsed_time(x1), world, dev)
    e2e_value = whole_job_value(flops, args.e2e_steps, world, e2e_ms)
    assert bool(torch.isfinite(hl).all()), "non-finite LSE in the end-to-end result"

    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    if rank != 0:
        return 0

    # The other workloads, timed after the headline in the same run (one GPU).
    per_config = None
    want = args.per_config == "on" or (args.per_config == "auto" and world == 1 and args.workload == DEFAULT_WORKLOAD
                                         and args.batch is None and args.seq is None and not args.noncausal
                                         and not bwd and splits == 1)
    if want:
        del hq, hk, hv, ho, hl
        e2e_step = ws_host = None   # drops the e2e step's device buffers
        torch.cuda.empty_cache()
        per_config = {}
        for name in PER_CONFIG:
            if name == w.name:
                continue
            per_config[name] = per_config_line(fa, name, dev, stream, peaks, sms, local_rank, warm=args.warm,
                                               cpu_baseline=not args.no_cpu_baseline)
            if name == "cross_b2_h8_m1000_n3000_d96_peaked":
                per_config[name + "+splitkv"] = per_config_line(fa, name, dev, stream, peaks, sms, local_rank,
                                                                splitkv=True, warm=args.warm)

    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    peak = float(peaks["bf16_tflops"])
    pspec, pspec_src = spec_peak(sms, mhz, BF16_FLOP_PER_CLK_SM, "bf16")
    bound, peak_source = "tensor", (f"{peaks.get('source')} bf16_tflops (burst); sustained "
                                    f"{peaks.get('bf16_tflops_sustained')}")
    frac_sust = achieved / float(peaks.get("bf16_tflops_sustained", peak))
    ach_scale = 1.0
    if x3:
        # Three TF32 products per matrix product: the tensor core executes 3x the attention
        # FLOPs, against the TF32 peak (measured bf16 x the nominal TF32 : BF16 ratio 1.1 : 2.25).
        ach_scale = 3.0
        achieved *= 3.0
        peak = float(peaks["bf16_tflops"]) * 1.1 / 2.25
        pspec, pspec_src = spec_peak(sms, mhz, TF32_FLOP_PER_CLK_SM, "tf32")
        peak_source = (f"{peaks.get('source')} bf16_tflops x 1.1/2.25 (nominal dense TF32 : BF16); achieved "
                       f"counts the 3 TF32 products per attention FLOP")
        frac_sust = achieved / (float(peaks.get("bf16_tflops_sustained", peak)) * 1.1 / 2.25)
    elif bwd and w.D in (64, 96, 128):
        # The tensor-core backward: achieved counts the algorithm's five products (its
        # kernels execute seven: S and dP are rebuilt in both the dK/dV and the dQ kernel).
        peak_source = (f"{peaks.get('source')} bf16_tflops (burst); achieved counts the 5 products of the "
                       f"recomputing backward (7 executed)")
    elif not bf16 or bwd:
        # The fp32 path and the backward run on the CUDA cores (fp32 FMA, no tensor cores):
        # its ceiling is SMs x 128 fp32 lanes x 2 FLOP per FMA x max SM clock.
        peak = sms * 128 * 2 * mhz * 1e6 / 1e12
        pspec, pspec_src = peak, f"derived: {sms} SMs x 128 fp32 lanes x 2 FLOP x {mhz:.0f} MHz (fp32 FMA)"
        bound = "alu"
        peak_source = pspec_src
        frac_sust = None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v_cpu, secs, nrows, cores, desc = oracle_sample(w, args.cpu_seconds)
        model, blas = host_cpu()
        cpu = {"value": v_cpu, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": secs, "cpu_model": model, "blas": blas}
    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": max_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32", "data": "synthetic",
        "config": dict(w.describe(), parallelism=f"replicas x{world}", kv_splits=splits,
                       **({"f32_path": "x3 (fa_fwd_f32x3)" if x3 else "ieee (fa_fwd_f32)"} if not bf16 else {}),
                       l2=l2),
        "pct_of_peak": 100.0 * value / world * ach_scale / peak,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak,
                     "traffic": (recorded_traffic(w.describe()["workload"]) if bf16 and splits == 1 and not bwd else
                                 recorded_traffic(w.describe()["workload"], "x3") if x3 else None),
                     "peak_source": peak_source,
                     "frac_of_sustained": frac_sust,
                     "peak_spec": pspec, "peak_spec_source": pspec_src, "frac_of_spec": achieved / pspec,
                     "launch_ms": ls["mean"], "launch_ms_median": ls["median"], "launch_ms_min": ls["min"],
                     "achieved_median": flops * ach_scale / (ls["median"] * 1e-3) / 1e12},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.e2e_steps, "steps": args.e2e_steps, "api": e2e_api},
        "gpu_launches": steps * (3 if bwd else (2 if splits > 1 or x3 else 1)),
        "clocks": clocks,
        "clocks_rejected": clocks_rejected(clocks),
    }
    if per_config is not None:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    from flashattention_fa_fwd_gb300.inputs import WORKLOADS

    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(WORKLOADS)}")
    w = WORKLOADS[args.workload]
    import dataclasses

    if args.batch is not None:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}_batch{args.batch}")
    if args.seq is not None:
        w = dataclasses.replace(w, M=args.seq, N=args.seq, name=f"{w.name}_seq{args.seq}")
    if args.noncausal:
        w = dataclasses.replace(w, causal=False, name=f"{w.name}_noncausal")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        return reference_arm(args, w, rank, world)
    return gpu_arm(args, w, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
