#!/usr/bin/env python3
"""Benchmark: causal bf16 prefill TFLOP/s (B4 H32 S2048 D128) and decode HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one attn_fwd call on the prefill workload (the headline `value`),
timed with CUDA events on the launching stream, L2 flushed between steps
outside the events.  The decode workload (B64 H32 D128, cache padded to 8192,
lengths uniform on [4096, 8192]) is timed the same way and reported under
"decode".  "e2e" is the same prefill through attn_fwd_host from pinned host
buffers, copies inside the timed call.  "configs" holds every workload --
the fp32 one (B2 H4 S128 D64), the headline, causal + key padding (B8 H16
S4096), long context (B1 H32 S16384) and decode -- each with its time, its
roofline and the fp64 CPU oracle timed on the host cores (in full for the
fp32, headline and decode workloads; on a seeded row sample, with an
extrapolated full time, for the padded and long ones).  The line's
`cpu_baseline` is the oracle over the whole headline workload.  Rank 0
prints one JSON line.

--impl reference times the fp64 CPU checker (the only reference this method
has) on a bounded sample of the same workload, on the host cores.

Profiling and extra runs (not part of the default line):
    --only prefill | decode        one kernel family
    --only decode-gqa [--decode-hkv 32,8,1]
                                   grouped-query decode on the decode workload's shape
    --only s-sweep                 prefill time against sequence length (S = 128 .. 65536)

Under torchrun (N > 1) each rank runs its own shard of the global batch
(sequences are independent problems: no data-path collective); the process
group carries only a barrier and the max over ranks of the timings.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from transformer_scaled_dot_fwd_gb300 import workloads as wl  # noqa: E402

METRIC = "causal attn fwd TFLOP/s (B4 H32 S2048 D128 bf16) and % peak; decode HBM GB/s"
L2_FLUSH_BYTES = 256 << 20   # > the 129 MB L2
SETTLE_S = 0.01              # untimed flush + call before the timed steps (see time_steps)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- counting

def prefill_flops(B, H, Sq, Skv, D, causal):
    """4*B*H*Sq*Skv*D (scores and weights @ V), halved for causal."""
    f = 4.0 * B * H * Sq * Skv * D
    return f / 2.0 if causal else f


def decode_bytes(H, D, kv_len, elem=2):
    """K and V bytes a decode step must read: sum_b 2*H*L_b*D*elem."""
    return float(sum(2.0 * H * float(L) * D * elem for L in kv_len))


def decode_flops(H, D, kv_len):
    return float(sum(4.0 * H * float(L) * D for L in kv_len))


# ----------------------------------------------------------------------------- environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        return dist
    return None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every PERIOD_MS milliseconds."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")
    PERIOD_MS = 20

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        """Start sampling and wait (up to 5 s) until the first sample is written."""
        self.window = None
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.file.name) == 0:
            time.sleep(0.01)

    def mark(self, t_begin, t_end):
        """Wall-clock bounds (time.time()) of the timed region."""
        self.window = (t_begin, t_end)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = []
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[9].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    float("0." + r[9].split(".")[1]) if "." in r[9] else 0.0
            except (ValueError, IndexError):
                ts = 0.0
            if self.window and self.window[0] - 0.02 <= ts <= self.window[1] + 0.02:
                inside.append(r)
        if inside:
            rows = inside
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": len(inside), "period_ms": self.PERIOD_MS}


# ----------------------------------------------------------------------------- timing

def time_steps(fn, steps, stream, flush, window=None):
    """Run fn() `steps` times; CUDA events on `stream` around each call, L2
    flushed between calls outside the events (untimed flush + call first,
    for SETTLE_S).  Returns per-step ms.  If `window` is a dict, its "t0" and
    "t1" receive the wall-clock times (time.time()) that bracket the timed
    steps, for the clock sampler.

    torch creates a CUDA event at its first record(); every event is recorded
    once before the loop, so that no event is created between a step's flush
    and its call (from an idle device that host work would otherwise show up
    as a gap inside the first timed step)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in starts + ends:
        e.record(stream)
    # untimed first: one flush + call (the flush kernel's first launch loads
    # its module, which on a fresh machine can take a quarter of a second),
    # then flush + call repeated for SETTLE_S, so that the timed steps do not
    # start on a device that has just dropped to its idle clocks
    flush()
    fn()
    torch.cuda.synchronize()
    t_settle = time.perf_counter()
    while time.perf_counter() - t_settle < SETTLE_S:
        flush()
        fn()
        torch.cuda.synchronize()
    if window is not None:
        window["t0"] = time.time()
    for s in range(steps):
        flush()
        starts[s].record(stream)
        fn()
        ends[s].record(stream)
    torch.cuda.synchronize()
    if window is not None:
        window["t1"] = time.time()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def kernel_source_digest(main="prefill_tc.cu"):
    """Short hash of a kernel's source files (the kernel file, ptx.cuh, kernels.h)."""
    h = hashlib.sha256()
    for f in (main, "ptx.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "transformer_scaled_dot_fwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(name, main):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_src = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_src and m_b) or m_src.group(1) != kernel_source_digest(main):
        return None
    return float(m_b.group(1))


# ----------------------------------------------------------------------------- CPU checker timing

def cpu_oracle_sample(q, k, v, w, kv_len, budget_s, rng_seed=0):
    """Time the fp64 checker on a random sample of rows of the workload; the
    sample is sized from a short calibration run to take about budget_s.
    Returns (TFLOP/s, description, threads)."""
    import oracle
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    kv_host = None if kv_len is None else kv_len.cpu().numpy()
    rng = np.random.default_rng(rng_seed)

    def rows_and_flops(n):
        b = rng.integers(0, w.B, n)
        h = rng.integers(0, w.H, n)
        i = rng.integers(0, w.S, n)
        vis = (i + 1) if w.causal else np.full(n, w.S)
        if kv_host is not None:
            L = kv_host[b]
            vis = np.where(i < L, np.minimum(vis, L), 0)
        return np.stack([b, h, i], 1), float(np.sum(4.0 * w.D * vis))

    rows, _ = rows_and_flops(256)
    t0 = time.perf_counter()
    oracle.attention_rows(qc, kc, vc, rows, scale=w.softmax_scale, causal=w.causal, kv_len=kv_host)
    per_row = max((time.perf_counter() - t0) / 256, 1e-7)
    n = int(min(max(budget_s / per_row, 256), w.B * w.H * w.S))
    rows, flops = rows_and_flops(n)
    t0 = time.perf_counter()
    oracle.attention_rows(qc, kc, vc, rows, scale=w.softmax_scale, causal=w.causal, kv_len=kv_host)
    dt = time.perf_counter() - t0
    desc = (f"{n} query rows of the {w.name} workload drawn uniformly with replacement "
            f"({flops / 1e9:.2f} GFLOP of the method's count), fp64, {dt:.1f} s")
    return flops / dt / 1e12, desc, threads, dt


def oracle_threads():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def visible_keys(w, kv_host, b, i):
    """Keys query row i of sequence b sees (0 for a padded query row)."""
    L = w.S if kv_host is None else int(kv_host[b])
    if i >= L:
        return 0
    return min(i + 1, L) if w.causal else L


def workload_flops(w, kv_host):
    """The method's count, as the GPU legs use it: 4*B*H*S*S*D, halved for
    causal; with key padding the effective count sum_b 4*H*L_b*L_b*D/2."""
    if kv_host is None:
        return prefill_flops(w.B, w.H, w.S, w.S, w.D, w.causal)
    return float(sum(4.0 * w.H * float(L) * float(L) * w.D / (2.0 if w.causal else 1.0) for L in kv_host))


def cpu_oracle_full(q, k, v, w, kv_len, repeat=1):
    """The fp64 oracle over the whole workload (every output row), timed on
    the host cores; the fastest of `repeat` runs."""
    import oracle
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    kv_host = None if kv_len is None else kv_len.cpu().numpy()
    best = None
    for _ in range(repeat):
        t0 = time.perf_counter()
        oracle.attention(qc, kc, vc, scale=w.softmax_scale, causal=w.causal, kv_len=kv_host)
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    flops = workload_flops(w, kv_host)
    rows = w.B * w.H * w.S
    return {"value": flops / best / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"the whole {w.name} workload: all {rows} output rows, fp64, {best:.3f} s"
                      + (f" (fastest of {repeat} runs)" if repeat > 1 else ""),
            "seconds": best, "rows_per_s": rows / best, "extrapolated": False}


def cpu_oracle_rows_sample(q, k, v, w, kv_len, seed):
    """The fp64 oracle on a seeded row sample: for every (b, h) the rows 0, 1,
    127, 128, L_b - 1, L_b and S - 1, plus 64 rows drawn without replacement.
    Reports the sample's TFLOP/s and rows/s, and a full-workload time
    extrapolated from the sample by the method's flop count."""
    import oracle
    kv_host = None if kv_len is None else kv_len.cpu().numpy()
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        L = w.S if kv_host is None else int(kv_host[b])
        fixed = {0, 1, 127, 128, L - 1, L, w.S - 1}
        for h in range(w.H):
            pick = {i for i in fixed if 0 <= i < w.S} | set(rng.choice(w.S, 64, replace=False).tolist())
            rows += [(b, h, i) for i in sorted(pick)]
    rows = np.array(rows, dtype=np.int64)
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    t0 = time.perf_counter()
    oracle.attention_rows(qc, kc, vc, rows, scale=w.softmax_scale, causal=w.causal, kv_len=kv_host)
    dt = time.perf_counter() - t0
    sample_flops = float(sum(4.0 * w.D * visible_keys(w, kv_host, int(b), int(i)) for b, _, i in rows))
    exact_flops = float(sum(4.0 * w.D * visible_keys(w, kv_host, b, i) for b in range(w.B) for i in range(w.S)) * w.H)
    rate = sample_flops / dt
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": (f"{len(rows)} query rows of the {w.name} workload (per (b, h): rows 0, 1, 127, 128, "
                       f"L-1, L, S-1 and 64 drawn without replacement, seed {seed}), fp64, {dt:.2f} s"),
            "seconds": dt, "rows": int(len(rows)), "rows_per_s": len(rows) / dt,
            "extrapolated": True, "extrapolated_full_seconds": exact_flops / rate}


def cpu_oracle_decode(q, kc, vc, kv_len, dwk):
    """The fp64 oracle over the whole decode workload (every (b, h) row),
    reported as GB/s of the K/V bytes the method reads and as TFLOP/s."""
    import oracle
    lens = kv_len.cpu().numpy()
    qh, kh, vh = q.cpu(), kc.cpu(), vc.cpu()
    t0 = time.perf_counter()
    oracle.decode(qh, kh, vh, kv_len=lens)
    dt = time.perf_counter() - t0
    nbytes = decode_bytes(dwk.H, dwk.D, lens.tolist())
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"the whole {dwk.name} workload: all {dwk.B * dwk.H} query rows, fp64, {dt:.3f} s",
            "seconds": dt, "tflops": decode_flops(dwk.H, dwk.D, lens.tolist()) / dt / 1e12,
            "extrapolated": False}


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = wl.PREFILL
    q, k, v, kv_len = wl.prefill_inputs(w, device="cpu")
    # about 150 s of checker time for the whole run, whatever --steps is (each
    # step a sample of at least 256 rows), at most 10 s a step
    per_step = max(0.01, min(10.0, 150.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        cpu_oracle_sample(q, k, v, w, kv_len, per_step / 4)
    vals, times, desc, threads = [], [], "", 0
    for s in range(args.steps):
        tf, desc, threads, dt = cpu_oracle_sample(q, k, v, w, kv_len, per_step, rng_seed=s + 1)
        vals.append(tf)
        times.append(dt)
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": float(np.mean(times) * 1e3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16-rounded inputs)",
        "config": config_dict(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_env(device, seeds):
    """Versions and seeds behind a measurement."""
    driver = None
    try:
        r = subprocess.run(["nvidia-smi", "-i", str(device.index or 0), "--query-gpu=driver_version",
                            "--format=csv,noheader"], capture_output=True, text=True, timeout=10)
        driver = r.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    return {"torch": torch.__version__, "cuda_runtime": torch.version.cuda, "driver": driver,
            "device": torch.cuda.get_device_name(device), "sms": torch.cuda.get_device_properties(device).multi_processor_count,
            "seeds": seeds}


def config_dict(w, world):
    return {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": w.causal,
            "global_batch": w.B * world, "seq_len": w.S,
            "parallelism": f"dp{world} (independent sequences per GPU, no collective)" if world > 1 else "single GPU",
            "l2": "flushed between steps (256 MB write), outside the timed events",
            "timing": "CUDA events on the launching stream around each call; sum over steps; max over ranks; "
                      "before the timed steps, untimed flush + call for 10 ms after the warm-up steps"}


def run_ours(args):
    import transformer_scaled_dot_fwd_gb300 as attn
    from transformer_scaled_dot_fwd_gb300 import build as _build

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    if rank == 0 or world == 1:
        _build.build(quiet=True)
    barrier(dist, device)
    attn.lib()
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def flush():
        flush_buf.fill_(1.0)

    peaks, peak_src = load_peaks()

    # -------------------------------------------------------------- prefill (headline)
    w = wl.PREFILL
    if args.only == "decode":
        return run_decode_only(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist)
    if args.only == "decode-gqa":
        return run_decode_gqa(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist)
    if args.only == "s-sweep":
        return run_s_sweep(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist)
    if args.only == "prefill-configs":
        return run_prefill_configs(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist)
    q, k, v, kv_len = wl.prefill_inputs(w, device=device, seed=w.seed + 1000 * rank)
    out = torch.empty_like(q)

    def step():
        attn.attn_fwd(q, k, v, out=out, scale=w.softmax_scale, causal=w.causal, kv_len=kv_len)

    # the clock sampler starts first (its first sample can take seconds), so
    # that the warm-up steps run right before the timed ones on a busy device
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    attn.attn_device_status()
    barrier(dist, device)
    torch.cuda.synchronize()
    window = {}
    ms = time_steps(step, args.steps, stream, flush, window)
    wall = window["t1"] - window["t0"]
    sampler.mark(window["t0"], window["t1"])
    clocks = sampler.stop()
    barrier(dist, device)
    attn.attn_device_status()
    total_ms = max_over_ranks(dist, float(sum(ms)), device)
    flops_step = prefill_flops(w.B, w.H, w.S, w.S, w.D, w.causal)
    value = world * flops_step * args.steps / (total_ms * 1e-3) / 1e12
    avg_ms = float(sum(ms)) / args.steps
    achieved = flops_step / (avg_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    traffic = profiled_traffic("prefill_tc_B4H32S2048D128.md", "prefill_tc.cu")
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} bf16 dense (burst: the kernel is timed alone)",
                # the same figure against the seconds-long, power-capped GEMM rate
                "peak_sustained": peak_sus, "frac_sustained": achieved / peak_sus,
                "kernel": "prefill_tc_kernel<128>",
                "algorithmic_flops_per_launch": flops_step}

    # -------------------------------------------------------------- decode
    decode, decode_tensors = (None, None) if args.only == "prefill" else decode_leg(
        args, attn, device, stream, flush, peaks, peak_src, world, rank, dist, keep=True)
    e2e = None if args.no_e2e else e2e_leg(args, attn, q, k, v, out, w, flops_step, world, dist, device)
    cpu_on = rank == 0 and world == 1 and not args.no_cpu_baseline
    cpu = cpu_oracle_full(q, k, v, w, kv_len) if cpu_on else None
    configs = None
    if args.only == "all" and not args.no_configs:
        configs = config_legs(args, attn, device, stream, flush, peaks, world, rank, dist, cpu_on)
        configs["prefill"] = {"workload": w.name, "seed": w.seed + 1000 * rank, "ms_per_step": avg_ms,
                              "TFLOP_per_s": achieved, "roofline": roofline, "cpu_baseline": cpu,
                              "note": "the headline workload: the line's own value"}
        if decode is not None:
            configs["decode"] = dict(decode)
            if cpu_on:
                configs["decode"]["cpu_baseline"] = cpu_oracle_decode(*decode_tensors, wl.DECODE)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V rounded to bf16)",
        "config": config_dict(w, world),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "decode": decode, "configs": configs,
        "step_ms": {"mean": avg_ms, "median": float(sorted(ms)[len(ms) // 2]), "min": float(min(ms)),
                    "max": float(max(ms))},
        "clocks": clocks, "gpu_launches": args.steps,
        "wall_s_timed_region": wall, "kernel_source_digest": kernel_source_digest(),
        "env": run_env(device, {"prefill": w.seed, "decode": wl.DECODE.seed, "rank_offset": 1000}),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def config_legs(args, attn, device, stream, flush, peaks, world, rank, dist, cpu_on):
    """The other workloads beside the headline one, each with its own time,
    roofline and fp64 oracle baseline: the fp32 workload (oracle run in
    full), the padded and the long-context workloads (oracle on a seeded row
    sample, with a full time extrapolated from it)."""
    out = {}
    for name in ("tiny_f32", "padded", "long"):
        line, (q, k, v, kv_len) = prefill_workload_leg(name, args, attn, device, stream, flush, peaks,
                                                       world, rank, dist)
        if cpu_on:
            w = wl.PREFILL_WORKLOADS[name]
            line["cpu_baseline"] = (cpu_oracle_full(q, k, v, w, kv_len, repeat=5) if name == "tiny_f32"
                                    else cpu_oracle_rows_sample(q, k, v, w, kv_len, seed=w.seed))
        out[name] = line
        del q, k, v, kv_len
        torch.cuda.empty_cache()
    return out


def decode_leg(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist, keep=False):
    dwk = wl.DECODE
    if args.decode_batch:
        dwk = wl.DecodeWorkload(dwk.name.replace("B64", f"B{args.decode_batch}"), args.decode_batch,
                                dwk.H, dwk.Skv, dwk.D, dwk.seed, dwk.kv_len_range)
    dq, dk, dv, dkl = wl.decode_inputs(dwk, device=device, seed=dwk.seed + 1000 * rank)
    dout = torch.empty_like(dq)

    def dstep():
        attn.attn_decode(dq, dk, dv, out=dout, kv_len=dkl)

    for _ in range(args.warmup):
        dstep()
    attn.attn_device_status()
    dms = time_steps(dstep, args.steps, stream, flush)
    attn.attn_device_status()
    dtotal = max_over_ranks(dist, float(sum(dms)), device)
    dbytes = decode_bytes(dwk.H, dwk.D, dkl.cpu().tolist())
    d_avg = float(sum(dms)) / args.steps
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    d_gbs = dbytes / (d_avg * 1e-3) / 1e9
    decode = {
        "workload": dwk.name, "seed": dwk.seed + 1000 * rank,
        "value": world * dbytes * args.steps / (dtotal * 1e-3) / 1e9,
        "unit": "GB/s", "ms_per_step": d_avg,
        "tflops": decode_flops(dwk.H, dwk.D, dkl.cpu().tolist()) / (d_avg * 1e-3) / 1e12,
        "splits_per_head": attn.attn_decode_splits(dwk.B, dwk.H, dwk.Skv, dwk.D),
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": d_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": d_gbs / hbm_peak,
                     "traffic": profiled_traffic("decode_partial_B64H32Skv8192D128.md", "decode.cu")
                     if not args.decode_batch else None,
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": dbytes},
    }
    if keep:
        return decode, (dq, dk, dv, dkl)
    del dq, dk, dv, dout
    return decode


def run_decode_gqa(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist):
    """Grouped-query decode on the decode workload's shape (B64 H32 D128, cache
    padded to 8192, lengths U{4096..8192}) for H_kv in {32, 8, 1}: time, the
    K/V bytes a step must read (sum_b 2*H_kv*L_b*D*2) and the flops (sum_b
    4*H*L_b*D), so that flops / bytes = H / H_kv -- the intensity the pages
    predict for grouped decode ('Attention from First Principles', section 6;
    Exercise F).  One JSON line per H_kv; not part of the default run."""
    dwk = wl.DECODE
    B = args.decode_batch or dwk.B
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    lens = wl.draw_lengths(B, dwk.kv_len_range, dwk.seed + 1000 * rank).tolist()
    kl = torch.tensor(lens, dtype=torch.int32, device=device)
    for H_kv in (args.decode_hkv or (dwk.H, 8, 1)):
        g = torch.Generator(device=device).manual_seed(dwk.seed + H_kv)
        q = torch.randn(B, dwk.H, dwk.D, device=device, generator=g).to(torch.bfloat16)
        kc = torch.randn(B, H_kv, dwk.Skv, dwk.D, device=device, generator=g).to(torch.bfloat16)
        vc = torch.randn(B, H_kv, dwk.Skv, dwk.D, device=device, generator=g).to(torch.bfloat16)
        out = torch.empty_like(q)

        def step():
            attn.attn_decode(q, kc, vc, out=out, kv_len=kl)

        for _ in range(args.warmup):
            step()
        attn.attn_device_status()
        ms = time_steps(step, args.steps, stream, flush)
        attn.attn_device_status()
        avg = max_over_ranks(dist, float(sum(ms)), device) / args.steps
        nbytes = decode_bytes(H_kv, dwk.D, lens)
        flops = decode_flops(dwk.H, dwk.D, lens)
        if rank == 0:
            print(json.dumps({
                "decode_gqa": {"workload": f"KV-cache decode B{B} H{dwk.H} H_kv{H_kv} D{dwk.D} Skv<={dwk.Skv} bf16",
                               "ms_per_step": avg, "bytes_per_step": nbytes, "flops_per_step": flops,
                               "intensity_flop_per_byte": flops / nbytes,
                               "GB_per_s": nbytes / (avg * 1e-3) / 1e9,
                               "hbm_frac": nbytes / (avg * 1e-3) / 1e9 / hbm_peak,
                               "TFLOP_per_s": flops / (avg * 1e-3) / 1e12}}), flush=True)
        del q, kc, vc, out
    if dist is not None:
        dist.destroy_process_group()
    return 0


PROFILE_SUMMARIES = {"prefill": "prefill_tc_B4H32S2048D128.md", "padded": "prefill_tc_padded_B8H16S4096D128.md",
                     "long": "prefill_tc_long_B1H32S16384D128.md", "tiny_f32": "prefill_f32_B2H4S128D64.md"}


def prefill_workload_leg(name, args, attn, device, stream, flush, peaks, world, rank, dist):
    """Time one prefill workload alone (CUDA events, L2 flushed between calls).
    Returns (line, (q, k, v, kv_len)).  FLOPs: the nominal count
    4*B*H*S*S*D/2 and, with key padding, the effective count
    sum_b 4*H*L_b*L_b*D/2 of the visible (query, key) pairs, which the
    fraction of peak uses.  The fp32 workload is latency-bound (16.8 MFLOP):
    it has no roofline, its figure is the time per call."""
    w = wl.PREFILL_WORKLOADS[name]
    q, k, v, kv_len = wl.prefill_inputs(w, device=device, seed=w.seed + 1000 * rank)
    out = torch.empty_like(q)

    def step():
        attn.attn_fwd(q, k, v, out=out, scale=w.softmax_scale, causal=w.causal, kv_len=kv_len)

    for _ in range(args.warmup):
        step()
    attn.attn_device_status()
    ms = time_steps(step, args.steps, stream, flush)
    attn.attn_device_status()
    avg = max_over_ranks(dist, float(sum(ms)), device) / args.steps
    nominal = prefill_flops(w.B, w.H, w.S, w.S, w.D, w.causal)
    effective = workload_flops(w, None if kv_len is None else kv_len.cpu().numpy())
    kernel = "prefill_f32_kernel" if w.dtype == "f32" else f"prefill_tc_kernel<{w.D}>"
    line = {"workload": w.name, "dtype": w.dtype, "seed": w.seed + 1000 * rank, "steps": args.steps,
            "ms_per_step": avg, "us_per_step": avg * 1e3,
            "flops_nominal": nominal, "flops_effective": effective,
            "TFLOP_per_s_nominal": nominal / (avg * 1e-3) / 1e12,
            "TFLOP_per_s_effective": effective / (avg * 1e-3) / 1e12,
            "kernel": kernel, "gpu_launches": args.steps,
            "step_ms": {"median": float(sorted(ms)[len(ms) // 2]), "min": float(min(ms)), "max": float(max(ms))}}
    if w.dtype == "f32":
        line["roofline"] = {"bound": "latency", "note": "16.8 MFLOP per call: too small to fill the GPU; "
                            "the figure is the time per call"}
    else:
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        achieved = line["TFLOP_per_s_effective"]
        peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        line["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                            "frac": achieved / peak, "peak_sustained": peak_sus,
                            "frac_sustained": achieved / peak_sus,
                            "traffic": profiled_traffic(PROFILE_SUMMARIES[name], "prefill_tc.cu"),
                            "kernel": kernel, "algorithmic_flops_per_launch": effective}
    return line, (q, k, v, kv_len)


def run_prefill_configs(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist):
    """The prefill workloads other than the headline one, each timed alone
    (see prefill_workload_leg).  One JSON line per workload; not part of the
    default run."""
    names = [args.prefill_config] if args.prefill_config else ["tiny_f32", "padded", "long"]
    for name in names:
        line, tensors = prefill_workload_leg(name, args, attn, device, stream, flush, peaks, world, rank, dist)
        if rank == 0:
            print(json.dumps({"prefill_config": line}), flush=True)
        del tensors
    if dist is not None:
        dist.destroy_process_group()
    return 0


def loglog_slope(xs, ys):
    """Least-squares slope of log(y) against log(x)."""
    lx, ly = np.log(np.asarray(xs, float)), np.log(np.asarray(ys, float))
    return float(np.polyfit(lx, ly, 1)[0]) if len(xs) >= 2 else None


def run_s_sweep(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist):
    """Prefill time against sequence length at fixed batch (B4 H32 D128 bf16),
    causal and not: 'Attention from First Principles', Exercises, D (time vs S
    on log-log axes, slope 2 for the score work; where a naive implementation
    runs out of memory), with the score-tensor sizes of its section 5 and
    'Scaled dot-product attention with masking', "The memory problem".

    For each S: CUDA-event time per call (L2 flushed between calls), TFLOP/s,
    and the bytes a materialising implementation needs for the (B, H, S, S)
    bf16 score tensor alone, against the device's memory.  This path holds
    no score tensor: its device memory is Q, K, V and O.  One JSON line per
    (S, causal), then a summary line with the log-log slopes; not part of the
    default run."""
    sh = wl.S_SWEEP_SHAPE
    B, H, D = sh["B"], sh["H"], sh["D"]
    total_mem = torch.cuda.get_device_properties(device).total_memory
    tflops_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    rows = {True: [], False: []}
    first_naive_oom = None
    for S in wl.S_SWEEP:
        q, k, v = wl.s_sweep_inputs(S, device, rank)
        out = torch.empty_like(q)
        qkvo = 4 * q.numel() * q.element_size()
        naive_scores = B * H * S * S * 2
        naive_fits = naive_scores + qkvo <= total_mem
        if not naive_fits and first_naive_oom is None:
            first_naive_oom = S
        for causal in (True, False):
            def step():
                attn.attn_fwd(q, k, v, out=out, causal=causal)

            flops = prefill_flops(B, H, S, S, D, causal)
            est_ms = flops / (0.8 * tflops_peak * 1e12) * 1e3 + 0.01
            steps = int(min(args.steps, max(3, math.ceil(300.0 / est_ms))))
            for _ in range(args.warmup):
                step()
            attn.attn_device_status()
            ms = time_steps(step, steps, stream, flush)
            attn.attn_device_status()
            avg = max_over_ranks(dist, float(sum(ms)), device) / steps
            rows[causal].append((S, avg))
            if rank == 0:
                print(json.dumps({"s_sweep": {
                    "workload": f"{'causal' if causal else 'non-causal'} prefill B{B} H{H} S{S} D{D} bf16",
                    "S": S, "causal": causal, "steps": steps, "ms_per_call": avg,
                    "flops_per_call": flops, "TFLOP_per_s": flops / (avg * 1e-3) / 1e12,
                    "frac_of_peak": flops / (avg * 1e-3) / 1e12 / tflops_peak,
                    "device_bytes_qkvo": qkvo, "naive_score_tensor_bytes": naive_scores,
                    "naive_fits_in_device_memory": bool(naive_fits)}}), flush=True)
        del q, k, v, out
        torch.cuda.empty_cache()
    if rank == 0:
        summary = {"device_memory_bytes": total_mem, "peak_tflops": tflops_peak, "peak_source": peak_src,
                   "first_S_where_naive_scores_exceed_memory": first_naive_oom,
                   "l2": "flushed between calls (256 MB write), outside the timed events"}
        for causal in (True, False):
            pts = rows[causal]
            key = "causal" if causal else "non_causal"
            summary[f"slope_{key}_all"] = loglog_slope([s for s, _ in pts], [t for _, t in pts])
            big = [(s, t) for s, t in pts if s >= 2048]
            summary[f"slope_{key}_S_ge_2048"] = loglog_slope([s for s, _ in big], [t for _, t in big])
        print(json.dumps({"s_sweep_summary": summary}), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_decode_only(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist):
    decode = decode_leg(args, attn, device, stream, flush, peaks, peak_src, world, rank, dist)
    if rank == 0:
        print(json.dumps({"decode": decode}), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def e2e_leg(args, attn, q, k, v, out, w, flops_step, world, dist, device):
    """The same prefill through attn_fwd_host: inputs and output in pinned
    host memory, the library copying each chunk of heads in, computing it and
    copying it out (overlapped) inside every timed call."""
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hout = torch.empty(q.shape, dtype=q.dtype).pin_memory()

    def e2e_step():
        attn.attn_fwd_host(hq, hk, hv, out=hout, scale=w.softmax_scale, causal=w.causal)

    e2e_steps = max(1, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist, device)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t0, device)
    h2d = 3 * q.numel() * q.element_size()
    d2h = out.numel() * out.element_size()
    e2e = {"value": world * flops_step * e2e_steps / e2e_s / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": 1e3 * e2e_s / e2e_steps,
           "timing": "wall clock around attn_fwd_host (pinned host buffers; copies in, attention, copy out "
                     "overlapped by chunks inside the call); each call returns with the result in host memory"}
    del hq, hk, hv, hout
    return e2e


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (fp32, padded, long context) in the default line")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "decode-gqa", "s-sweep", "prefill-configs"],
                    default="all", help="profiling runs: time one kernel family only; s-sweep times "
                    "prefill against sequence length; prefill-configs times the other prefill workloads")
    ap.add_argument("--prefill-config", choices=["tiny_f32", "padded", "long"], default=None,
                    help="prefill-configs runs: one workload only")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="profiling runs: smaller decode batch than the workload's 64")
    ap.add_argument("--decode-hkv", type=lambda x: [int(v) for v in x.split(",")], default=None,
                    help="decode-gqa runs: comma-separated key/value head counts (default 32,8,1)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
