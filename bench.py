"""Throughput benchmark for exact tiled attention on GB300.

One step = one forward + one backward pass (all stages of the hot path)
over the Llama-shaped causal workload B=2 H=32 N=8192 d=128 (default; g4 is
its grouped-query form with 8 K/V heads), bf16 inputs
drawn from the seeded generator. Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c4|c2|c5|c3|c1|g4|s1|s2|d1|d2]

Under torchrun each rank runs its own replica of the workload on its own GPU
(the path shards by independent heads; there is no data exchange), timing
is max-over-ranks, and ``value`` is the whole-job FLOP rate.

``--impl reference`` times the fp64 CPU oracle as it stands on the host
cores, one bounded sample (one head's forward + backward) per step.

``--workload s1|s2`` instead times the standalone row softmax kernels (the
two-pass online form against the three-pass safe form) and reports GB/s;
``--workload d1`` times one paged-KV decode step and reports K/V GB/s (``d2``:
the same step with one-token cache blocks).
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "attention TFLOP/s (fwd; fwd+bwd) on 1 GB300 and % of dense BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def flops(w, direction):
    pairs = w.N * (w.N + 1) // 2 if True in w.causal else w.N * w.N
    per_pair = {"fwd": 4 * w.d, "bwd": 10 * w.d}[direction]
    return per_pair * w.B * w.H * pairs


def barrier(dist):
    """Line the ranks up (no-op at world size 1)."""
    if dist is not None:
        dist.barrier()


def max_over_ranks(values, dist, device):
    """Each value's maximum over the ranks: the slowest rank's time sets
    the job's time. The values themselves at world size 1."""
    values = [float(x) for x in values]
    if dist is None:
        return values
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank, world, ms):
    """Units per second over the whole job: every rank runs the same
    workload on its own GPU (weak scaling) and `ms` is the max-over-ranks
    time of one step."""
    return units_per_rank * world / (ms * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None, period_ms=20):
        self.bus_id = bus_id
        self.period_ms = period_ms
        self.proc = None
        self.lines = []          # (arrival time, line)
        self.thread = None
        self.t0 = self.t1 = None

    def __enter__(self):
        """Start sampling and wait (at most 5 s) for the first sample, so that
        the sampler is live when the timed region begins."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={self.period_ms}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def region_start(self):
        self.t0 = time.monotonic()

    def region_end(self):
        """Call after the timed region's final synchronize. Waits up to two
        periods for a sample taken after the region (used only when the
        region is shorter than the sampling period)."""
        self.t1 = time.monotonic()
        deadline = self.t1 + 2.5 * self.period_ms / 1000.0
        while (self.proc is not None and time.monotonic() < deadline
               and not any(t > self.t1 for t, _ in self.lines)):
            time.sleep(0.005)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        lines = list(self.lines)
        where = "all"
        if self.t0 is not None and self.t1 is not None:
            inside = [(t, l) for t, l in lines if self.t0 <= t <= self.t1]
            if inside:
                lines, where = inside, "timed region"
            else:
                after = [(t, l) for t, l in lines if t > self.t1][:1]
                lines, where = after, "first sample after the timed region (shorter than the period)"
        rows = []
        for _, line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.bus_id and parts[1].lower()[-12:] != self.bus_id.lower()[-12:]:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        smax = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        under_load = [s for s in sm if smax and s >= 0.3 * max(smax)] or sm
        return {"sm_mhz": statistics.median(under_load) if under_load else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "sampled": where,
                "power_w_max": max((num(r[4]) or 0.0) for r in rows)}


# -------------------------------------------------------------- oracle leg

def oracle_sample(w, q, k, v, do, heads, n=None, keep_first=False):
    """Time the fp64 oracle's forward + backward on the given heads, each
    restricted to its first n queries and keys (all N when n is None: a
    prefix of a head is itself a complete attention problem of length n).
    Returns (seconds, algorithmic FLOPs of the sample), plus the first
    head's oracle results {o, lse, dq, dk, dv} when keep_first is set."""
    from exact_tiled_attention_24_gb300.workloads import to_f64
    from oracle import attention_bwd_head, attention_fwd_head
    causal = True in w.causal
    n = w.N if n is None else n
    first = None
    t0 = time.perf_counter()
    for (b, h) in heads:
        hk = h // (w.H // w.kv_heads)  # the K/V head query head h reads
        qq, dd = to_f64(q[b, h, :n]), (to_f64(do[b, h, :n]) if do is not None else None)
        kk, vv = to_f64(k[b, hk, :n]), to_f64(v[b, hk, :n])
        fo = attention_fwd_head(qq, kk, vv, w.scale, causal)
        bo = attention_bwd_head(qq, kk, vv, dd, w.scale, causal) if do is not None else None
        if keep_first and first is None:
            first = {"o": fo[0], "lse": fo[1]}
            if bo is not None:
                first.update({"dq": bo[0], "dk": bo[1], "dv": bo[2]})
    dt = time.perf_counter() - t0
    pairs = n * (n + 1) // 2 if causal else n * n
    per_head = (4 * w.d + (10 * w.d if do is not None else 0)) * pairs
    if keep_first:
        return dt, per_head * len(heads), first
    return dt, per_head * len(heads)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def oracle_errors(first, gpu, b, h, G):
    """Max-abs and mean-abs difference between the GPU's outputs for head
    (b, h) and the oracle's. dk and dv are compared only with one K/V head
    per query head (with grouped heads the GPU's dk, dv sum over the group)."""
    import numpy as np
    out = {}
    for name, ref in first.items():
        if name in ("dk", "dv") and G != 1:
            continue
        t = gpu[name][b, h] if name not in ("dk", "dv") else gpu[name][b, h // G]
        got = t.detach().to("cpu", dtype=__import__("torch").float64).numpy()
        diff = np.abs(got - ref)
        out[name] = {"max_abs": float(diff.max()), "mean_abs": float(diff.mean())}
    return out


def run_reference(args, w, rank):
    if rank != 0:
        return None
    from exact_tiled_attention_24_gb300.workloads import workload_inputs
    q, k, v, *rest = workload_inputs(args.workload, with_do=True)
    do = rest[0] if rest else None
    heads = [(0, 0)]
    # One head per step for up to 30 steps; beyond that, each step takes the
    # head's first n queries and keys with n shrunk so that the whole run
    # costs about as much as 30 full-head steps (the rate is per FLOP).
    n = w.N if args.steps <= 30 else max(128, int(w.N * (30 / args.steps) ** 0.5) // 128 * 128)
    n = min(n, w.N)
    oracle_sample(w, q, k, v, do, heads, n)  # one untimed call (BLAS thread start-up)
    times, fl = [], 0
    for _ in range(args.steps):
        dt, fl = oracle_sample(w, q, k, v, do, heads, n)
        times.append(dt)
    total = sum(times)
    value = fl * args.steps / total / 1e12
    part = "" if n == w.N else f" (its first {n} queries and keys)"
    sample = (f"one head (b=0,h=0){part} of {args.workload} forward"
              f"{'+backward' if do is not None else ''} per step, fp64 NumPy oracle")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(args, w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def config_dict(args, w):
    kvh = "" if w.kv_heads == w.H else f" Hkv={w.kv_heads}"
    in_mb = (2 * w.H + 2 * w.kv_heads) * w.B * w.N * w.d * 2 // 2**20
    return {"workload": f"{w.name}: B={w.B} H={w.H}{kvh} N={w.N} d={w.d} causal={True in w.causal} bf16",
            "B": w.B, "H": w.H, "Hkv": w.kv_heads, "N": w.N, "d": w.d, "causal": True in w.causal,
            "directions": list(w.directions),
            "l2": "inputs larger than L2 (q,k,v,dO = %d MB vs 129 MB L2); no flush" % in_mb,
            "parallelism": f"replicas x{args.gpus} (independent heads per GPU, no collective)"}


# -------------------------------------------------------------- GPU leg

def traffic_for(kernel_key, sources):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    ent = data.get(kernel_key)
    if not ent:
        return None
    h = hashlib.sha256()
    for s in sources:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    if ent.get("source_sha256") != h.hexdigest():
        return None
    return ent.get("dram_bytes_per_launch")


def pick_peak(peaks, region_s, clocks):
    """The bf16 denominator for a kernel timed in this run: the burst figure
    for a timed region under a second that kept its clocks (no power cap),
    else the sustained figure (measured over seconds under the power cap)."""
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    name = "bf16_tflops" if region_s < 1.0 and not capped else "bf16_tflops_sustained"
    return float(peaks.get(name, FALLBACK_PEAKS[name])), name


def long_context_leg(args, dev, dist, peaks, peak_kind):
    """The long-context forward (B=1 H=16 N=32768 d=128, causal, q ~ N(0, 4^2))
    timed on its own with CUDA events, with its own clock samples."""
    import torch

    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300.workloads import WORKLOADS, workload_inputs

    w5 = WORKLOADS["c5"]
    q, k, v = (t.to(dev) for t in workload_inputs("c5", with_do=False)[:3])
    o = torch.empty_like(q)
    lse = torch.empty((w5.B, w5.H, w5.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(5, min(args.steps, 20))
    for _ in range(args.warmup):
        fa.fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(bus_id=bus) as clk:
        clk.region_start()
        e0.record(stream)
        for _ in range(steps):
            fa.fwd(q, k, v, causal=True, out=o, lse=lse)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clk.region_end()
    if fa.last_device_error(dev) != 0:
        raise RuntimeError("device error during the long-context forward")
    ms, = max_over_ranks([e0.elapsed_time(e1) / steps], dist, dev)
    clocks = clk.summary()
    peak, peak_name = pick_peak(peaks, ms * steps / 1e3, clocks)
    tflops = flops(w5, "fwd") / (ms * 1e-3) / 1e12
    fsrc = ["exact_tiled_attention_24_gb300/csrc/fa_fwd.cu", "exact_tiled_attention_24_gb300/csrc/fa_ptx.cuh"]
    return {"workload": "c5: B=1 H=16 N=32768 d=128 causal=True bf16, q ~ N(0, 4^2)", "steps": steps,
            "ms": ms, "tflops": tflops, "frac": tflops / peak, "peak": peak,
            "peak_source": f"{peak_kind} {peak_name}", "nominal_2250": tflops / 2250.0,
            "traffic": traffic_for("fwd_c5", fsrc), "clocks": clocks, "gpu_launches": steps}


def run_ours(args, w, rank, world, dist):
    import torch

    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300 import build as fabuild
    from exact_tiled_attention_24_gb300.workloads import workload_inputs

    fabuild.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    causal = True in w.causal
    has_bwd = "bwd" in w.directions
    q, k, v, *rest = workload_inputs(args.workload, with_do=has_bwd)
    do = rest[0] if rest else None
    host = [t.pin_memory() for t in (q, k, v) + ((do,) if do is not None else ())]
    qg, kg, vg = (t.to(dev) for t in host[:3])
    dog = host[3].to(dev) if has_bwd else None
    B, H, N, d = w.shape
    o = torch.empty_like(qg)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if has_bwd:
        dq, dk, dv = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
        Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # The backward in the order fa_bwd takes for this shape: the dQ sweep
    # forming D, then the dK/dV sweep; or the D pass, dK/dV, then dQ (one
    # stream here, so each kernel is timed on its own).
    fuse_d = has_bwd and fa.bwd_fuses_d(B, H, kg.shape[1], N, d)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fwd(qg, kg, vg, causal=causal, out=o, lse=lse)
        if ev is not None:
            ev[1].record(stream)
        if has_bwd and fuse_d:
            if ev is not None:
                ev[2].record(stream)  # no D pass
            fa.bwd_dq_d(qg, kg, vg, o, dog, lse, Dvec, dq, causal=causal)
            if ev is not None:
                ev[3].record(stream)
            fa.bwd_dkdv(qg, kg, vg, dog, lse, Dvec, dk, dv, causal=causal)
            if ev is not None:
                ev[4].record(stream)
        elif has_bwd:
            fa.bwd_preprocess(o, dog, Dvec)
            if ev is not None:
                ev[2].record(stream)
            fa.bwd_dkdv(qg, kg, vg, dog, lse, Dvec, dk, dv, causal=causal)
            if ev is not None:
                ev[3].record(stream)
            fa.bwd_dq(qg, kg, vg, dog, lse, Dvec, dq, causal=causal)
            if ev is not None:
                ev[4].record(stream)

    launches_per_step = (3 if fuse_d else 4) if has_bwd else 1
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.last_device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        bus = None
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(bus_id=bus) as clk:
        clk.region_start()
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clk.region_end()
    barrier(dist)
    elapsed_ms = t_start.elapsed_time(t_end)
    if fa.last_device_error(dev) != 0:
        raise RuntimeError("device error during the timed region")
    elapsed_ms, = max_over_ranks([elapsed_ms], dist, dev)

    # Distribution of the per-step device time (first kernel start to last
    # kernel end of each timed step).
    last = 4 if has_bwd else 1
    per_step = sorted(e[0].elapsed_time(e[last]) for e in evs)

    def pct(q):
        return per_step[min(len(per_step) - 1, int(q * (len(per_step) - 1) + 0.5))]

    step_stats = {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9), "n": len(per_step)}
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    if has_bwd:
        pre_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        k_a = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
        k_b = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
        dq_ms, dkdv_ms = (k_a, k_b) if fuse_d else (k_b, k_a)
    F_fwd = flops(w, "fwd")
    F_bwd = flops(w, "bwd") if has_bwd else 0
    F_step = F_fwd + F_bwd
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(F_step, world, ms_per_step) / 1e12
    peaks, peak_kind = load_peaks()

    # Dominant kernel: the one with the largest share of the step. Its
    # algorithmic FLOPs (the method's products it performs, 2mkn each):
    # fwd 4·d per pair (QKᵀ, PV); dkdv 8·d (recomputed Sᵀ, dPᵀ, dV, dK);
    # dq 2·d (dQ; its second recomputation of S and dP is not counted).
    bsrc = ["exact_tiled_attention_24_gb300/csrc/fa_bwd.cu", "exact_tiled_attention_24_gb300/csrc/fa_ptx.cuh"]
    fsrc = ["exact_tiled_attention_24_gb300/csrc/fa_fwd.cu", "exact_tiled_attention_24_gb300/csrc/fa_ptx.cuh"]
    cands = [("fwd", fwd_ms, F_fwd, fsrc)]
    if has_bwd:
        cands += [("bwd_dkdv", dkdv_ms, F_fwd * 2, bsrc), ("bwd_dq", dq_ms, F_fwd // 2, bsrc)]
    dom, dom_ms, dom_flops, srcs = max(cands, key=lambda c: c[1])
    clocks = clk.summary()
    region_s = elapsed_ms / 1e3
    peak, peak_name = pick_peak(peaks, region_s, clocks)
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} {peak_name}",
                "timed_region_s": region_s, "sm_mhz_median": clocks.get("sm_mhz"),
                "traffic": traffic_for(f"{dom}_{args.workload}", srcs)}

    # End-to-end: host buffers in, results out, every step, through the
    # library's host entry point (copies of one slice of heads overlap the
    # kernels of another). With --e2e-inflight 2 (the default) consecutive
    # steps alternate between two streams, each with its own device buffers
    # and host outputs (double buffering, as a training or serving loop would
    # run it), so one step's result copies overlap the next step's input
    # copies; every step still copies all of its inputs in and its results
    # out inside the timed region.
    e2e_steps = max(12, args.steps // 4)  # enough that the in-flight pipeline's start weighs little
    inflight = max(1, args.e2e_inflight)

    def host_out(t):
        return torch.empty(t.shape, dtype=t.dtype).pin_memory()

    sets = []
    for i in range(inflight):
        if i == 0:
            db = {"q": qg, "k": kg, "v": vg, "o": o, "lse": lse}
            if has_bwd:
                db.update({"dO": dog, "dq": dq, "dk": dk, "dv": dv})
            ws = Dvec if has_bwd else None
        else:
            db = {n: torch.empty_like(t) for n, t in (("q", qg), ("k", kg), ("v", vg), ("o", o), ("lse", lse))}
            if has_bwd:
                db.update({n: torch.empty_like(t) for n, t in (("dO", dog), ("dq", dq), ("dk", dk), ("dv", dv))})
            ws = torch.empty_like(Dvec) if has_bwd else None
        hb = {"q": host[0], "k": host[1], "v": host[2], "o": host_out(o), "lse": host_out(lse)}
        if has_bwd:
            hb["dO"] = host[3]
            for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
                hb[n] = host_out(t)
        st = stream if i == 0 else torch.cuda.Stream(dev)
        sets.append((hb, db, ws, st))
    hb0 = sets[0][0]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(hb0[n].numel() * hb0[n].element_size() for n in ("o", "lse", "dq", "dk", "dv") if n in hb0)

    def e2e_step(i):
        hb, db, ws, st = sets[i % inflight]
        with torch.cuda.stream(st):
            if has_bwd:
                fa.fwd_bwd_host(hb, db, ws, causal=causal, n_chunks=args.host_chunks)
            else:
                fa.fwd_host(hb, db, causal=causal, n_chunks=args.host_chunks)

    for i in range(2 * inflight):
        e2e_step(i)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    for _, _, _, st in sets[1:]:
        st.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    for _, _, _, st in sets[1:]:
        stream.wait_stream(st)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    if fa.last_device_error(dev) != 0:
        raise RuntimeError("device error during the end-to-end steps")
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    e2e_ms, = max_over_ranks([e2e_ms], dist, dev)
    e2e_value = whole_job_rate(F_step, world, e2e_ms) / 1e12
    if inflight > 1:  # every in-flight set computed the same results
        for n in ("o", "lse", "dq", "dk", "dv"):
            if n in sets[0][0] and not torch.equal(sets[0][0][n], sets[1][0][n]):
                raise RuntimeError(f"end-to-end steps disagree on {n}")

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(args, w),
        "step_ms": step_stats,
        "fwd_tflops": F_fwd / (fwd_ms * 1e-3) / 1e12,
        "fwd_ms": fwd_ms,
        "frac_of_peak": {"fwd_bwd": value / world / peak, "fwd": F_fwd / (fwd_ms * 1e-3) / 1e12 / peak,
                         "peak_tflops": peak, "peak_source": f"{peak_kind} {peak_name}",
                         "nominal_2250": value / world / 2250.0},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "host_chunks": args.host_chunks or "library default",
                "steps_in_flight": inflight},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
    }
    if args.workload == "c4" and not args.no_c5:
        result["c5_fwd"] = long_context_leg(args, dev, dist, peaks, peak_kind)
    if has_bwd:
        result["bwd_ms"] = {"preprocess": pre_ms, "dkdv": dkdv_ms, "dq": dq_ms}
        result["bwd_order"] = ("dq sweep forming D, then dkdv (no D pass)" if fuse_d
                               else "D pass, dkdv, dq")
        result["bwd_tflops"] = F_bwd / ((pre_ms + dkdv_ms + dq_ms) * 1e-3) / 1e12
        result["mfu_style_tflops"] = 3 * F_fwd * world / (ms_per_step * 1e-3) / 1e12
    if rank == 0 and not args.no_cpu_baseline:
        heads = [(0, 0)]
        dt, fl, first = oracle_sample(w, q, k, v, do, heads, keep_first=True)
        reps = 1  # heads timed: at least ~10 s of oracle work in all, at most 16 heads
        while dt < 10.0 and reps < 16:
            dt2, _ = oracle_sample(w, q, k, v, do, [(0, reps % w.H)])
            dt += dt2
            reps += 1
        gpu_out = {"o": o, "lse": lse}
        if has_bwd:
            gpu_out.update({"dq": dq, "dk": dk, "dv": dv})
        result["cpu_baseline"] = {
            "value": fl * reps / dt / 1e12, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{reps} head(s) of {args.workload} forward{'+backward' if has_bwd else ''}, "
                      f"fp64 NumPy oracle, {dt:.1f} s",
            "error_vs_gpu": {"head": "b=0 h=0 (the GPU's outputs of the last timed step)",
                             **oracle_errors(first, gpu_out, 0, 0, w.H // w.kv_heads)}}
    return result


# ------------------------------------------------- standalone row softmax

SOFTMAX_METRIC = "row softmax GB/s (x read once + y written once), online two-pass vs safe three-pass"


def run_softmax(args, rw, rank, world, dist):
    """Time the two-pass (online) and three-pass (safe) row softmax kernels on
    the same rows; value = online GB/s of algorithmic bytes (8 per element)."""
    import torch

    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300 import build as fabuild
    from exact_tiled_attention_24_gb300.workloads import make_rows

    fabuild.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    x_host = make_rows(rw.rows, rw.n, rw.seed, rw.std).pin_memory()
    x = x_host.to(dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    fns = {"online": fa.softmax_online, "safe": fa.softmax_safe}
    for fn in fns.values():
        for _ in range(args.warmup):
            fn(x, out=y)
    torch.cuda.synchronize(dev)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    barrier(dist)
    ms = {}
    with ClockSampler(bus_id=bus) as clk:
        clk.region_start()
        for name, fn in fns.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn(x, out=y)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms[name] = e0.elapsed_time(e1) / args.steps
        clk.region_end()
    barrier(dist)
    m_on, m_safe = max_over_ranks([ms["online"], ms["safe"]], dist, dev)
    ms = {"online": m_on, "safe": m_safe}
    alg_bytes = 8 * rw.rows * rw.n
    gbs = {k: alg_bytes / (v * 1e-3) / 1e9 for k, v in ms.items()}
    peaks, peak_kind = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    src = ["exact_tiled_attention_24_gb300/csrc/fa_softmax.cu", "exact_tiled_attention_24_gb300/csrc/fa_ptx.cuh"]
    # end to end through the host-memory call: pinned x to the device,
    # softmax, y back to pinned memory, slices of rows pipelined
    y_host = torch.empty_like(x_host).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 5))
    fa.softmax_host(x_host, y_host, x, y, online=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(e2e_steps):
        fa.softmax_host(x_host, y_host, x, y, online=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms, = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], dist, dev)
    res = {
        "metric": SOFTMAX_METRIC, "value": gbs["online"] * world, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms["online"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{rw.name}: softmax rows={rw.rows} n={rw.n} fp32, x ~ N(0, {rw.std:g}^2)",
                   "l2": "x and y %d MB each vs 129 MB L2; no flush" % (4 * rw.rows * rw.n // 2**20)},
        "safe_gbs": gbs["safe"], "safe_ms": ms["safe"],
        "speedup_online_vs_safe": ms["safe"] / ms["online"],
        "pages_claim": "1.33x nominal (4 vs 3 memory accesses per element), about 1.3x measured",
        "roofline": {"kernel": "softmax_online", "bound": "hbm", "achieved": gbs["online"], "peak": hbm,
                     "unit": "GB/s", "frac": gbs["online"] / hbm,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": traffic_for(f"softmax_online_{rw.name}", src)},
        "clocks": clk.summary(),
        "e2e": {"value": alg_bytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s",
                "h2d_bytes_per_step": 4 * rw.rows * rw.n, "d2h_bytes_per_step": 4 * rw.rows * rw.n,
                "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import softmax_safe
        k = 16
        xs = x_host[:k].to(torch.float64).numpy()
        reps, t0 = 0, time.perf_counter()
        while reps < 2000 and (reps == 0 or time.perf_counter() - t0 < 10.0):
            softmax_safe(xs)
            reps += 1
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": 8 * k * rw.n * reps / dt / 1e9, "unit": "GB/s", "cores": host_cores(),
                               "kind": "oracle",
                               "sample": f"{k} rows of {rw.name}, {reps} calls, fp64 NumPy oracle, {dt:.2f} s"}
    return res


def run_softmax_reference(args, rw, rank):
    if rank != 0:
        return None
    from exact_tiled_attention_24_gb300.workloads import make_rows
    from oracle import softmax_safe
    k = 16
    xs = make_rows(k, rw.n, rw.seed, rw.std).to(__import__("torch").float64).numpy()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        softmax_safe(xs)
        times.append(time.perf_counter() - t0)
    value = 8 * k * rw.n * args.steps / sum(times) / 1e9
    return {"impl": "reference", "metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{rw.name}: softmax rows={rw.rows} n={rw.n} fp32"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
                             "sample": f"{k} rows of {rw.name} per step, fp64 NumPy oracle"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# -------------------------------------------------------- paged-KV decode

DECODE_METRIC = "paged-KV decode GB/s (K and V bytes read per step)"


def decode_oracle_sample(dw, k=2):
    """The first k requests of a decode workload, drawn on the CPU by the
    same generator (same heads, block size and context-length range), as
    fp64 arrays for the oracle, with their K/V bytes."""
    import torch

    from exact_tiled_attention_24_gb300.workloads import DecodeWorkload, make_decode
    sw = DecodeWorkload(dw.name, k, dw.H, dw.Hkv, dw.d, dw.block_size, dw.min_len, dw.max_len, dw.n_splits,
                        dw.seed)
    q, kc, vc, table, lens = make_decode(sw, torch.device("cpu"))
    qs, kcs, vcs = (t.double().numpy() for t in (q, kc, vc))
    return qs, kcs, vcs, table.numpy(), lens.numpy(), int(lens.sum()) * dw.Hkv * dw.d * 4, k


def run_decode_reference(args, dw, rank):
    """The fp64 oracle's decode on a bounded sample of the workload: the
    first k requests drawn by the same generator (same heads, block size and
    context-length range), K/V bytes of the sample ÷ time."""
    if rank != 0:
        return None
    from oracle import decode_paged
    qs, kcs, vcs, tab, ln, sample_bytes, k = decode_oracle_sample(dw)
    decode_paged(qs, kcs, vcs, tab, ln, dw.d ** -0.5)  # one untimed call
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        decode_paged(qs, kcs, vcs, tab, ln, dw.d ** -0.5)
        times.append(time.perf_counter() - t0)
    value = sample_bytes * args.steps / sum(times) / 1e9
    return {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{dw.name}: decode B={dw.B} H={dw.H} Hkv={dw.Hkv} d={dw.d} "
                                   f"block={dw.block_size} context {dw.min_len}-{dw.max_len} "
                                   f"splits={dw.n_splits}"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
                             "sample": f"{k} requests of {dw.name} ({sample_bytes // (dw.Hkv * dw.d * 4)} "
                                       "tokens) per step, fp64 NumPy oracle"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_decode(args, dw, rank, world, dist):
    """Time one decode step (partial kernel + merge) over the resident cache;
    value = K/V bytes the step must read ÷ its time."""
    import torch

    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300 import build as fabuild
    from exact_tiled_attention_24_gb300.workloads import make_decode

    fabuild.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    q, kc, vc, table, lens = make_decode(dw, dev)
    ws = torch.empty(fa.decode_workspace_bytes(dw.B, dw.H, dw.d, dw.n_splits), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((dw.B, dw.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.decode_paged(q, kc, vc, table, lens, n_splits=dw.n_splits, workspace=ws, out=o, lse=lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.last_device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(bus_id=bus) as clk:
        clk.region_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clk.region_end()
    ms = e0.elapsed_time(e1) / args.steps
    if fa.last_device_error(dev) != 0:
        raise RuntimeError("device error during the timed region")
    barrier(dist)
    ms, = max_over_ranks([ms], dist, dev)
    tokens = int(lens.sum().item())
    kv_bytes = tokens * dw.Hkv * dw.d * 2 * 2
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    src = ["exact_tiled_attention_24_gb300/csrc/fa_decode.cu", "exact_tiled_attention_24_gb300/csrc/fa_ptx.cuh"]
    # end to end: q, table and lengths from pinned host memory, o and lse back
    hq, ht, hl = (t.cpu().pin_memory() for t in (q, table, lens))
    ho, hlse = torch.empty_like(o, device="cpu").pin_memory(), torch.empty_like(lse, device="cpu").pin_memory()
    e2e_steps = max(1, min(args.steps, 20))
    e0.record(stream)
    for _ in range(e2e_steps):
        q.copy_(hq, non_blocking=True)
        table.copy_(ht, non_blocking=True)
        lens.copy_(hl, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms, = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], dist, dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, ht, hl))
    d2h = ho.numel() * ho.element_size() + hlse.numel() * hlse.element_size()
    res = {
        "metric": DECODE_METRIC, "value": gbs * world, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{dw.name}: decode B={dw.B} H={dw.H} Hkv={dw.Hkv} d={dw.d} "
                               f"block={dw.block_size} context {dw.min_len}-{dw.max_len} "
                               f"(total {tokens} tokens) splits={dw.n_splits}",
                   "l2": "K/V %d MB read per step vs 129 MB L2; no flush" % (kv_bytes // 2**20)},
        "roofline": {"kernel": "decode_mma", "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": traffic_for(f"decode_mma_{dw.name}", src)},
        "clocks": clk.summary(),
        "e2e": {"value": kv_bytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": (2 if dw.n_splits > 1 else 1) * args.steps,  # kernel (+ merge)
    }
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import decode_paged
        qs, kcs, vcs, tab, ln, sample_bytes, k = decode_oracle_sample(dw)
        reps, t0 = 0, time.perf_counter()
        while reps < 400 and (reps == 0 or time.perf_counter() - t0 < 10.0):
            decode_paged(qs, kcs, vcs, tab, ln, dw.d ** -0.5)
            reps += 1
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": sample_bytes * reps / dt / 1e9, "unit": "GB/s", "cores": host_cores(),
                               "kind": "oracle",
                               "sample": f"{k} requests of {dw.name} drawn by the same generator, "
                                         f"{reps} calls, fp64 NumPy oracle, {dt:.2f} s"}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-c5", action="store_true",
                    help="skip the long-context forward leg of the default (c4) run")
    ap.add_argument("--e2e-inflight", type=int, default=2,
                    help="end-to-end steps in flight on their own streams and buffers (1: one after another)")
    ap.add_argument("--host-chunks", type=int, default=0,
                    help="slices of the end-to-end host pipeline (0: the library's choice)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from exact_tiled_attention_24_gb300.workloads import DECODE_WORKLOADS, ROW_WORKLOADS, WORKLOADS
    rw = ROW_WORKLOADS.get(args.workload)
    dw = DECODE_WORKLOADS.get(args.workload)
    w = WORKLOADS[args.workload] if rw is None and dw is None else None
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference" and dw is not None:
        res = run_decode_reference(args, dw, rank)
    elif args.impl == "reference":
        res = run_reference(args, w, rank) if rw is None else run_softmax_reference(args, rw, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
        if dw is not None:
            res = run_decode(args, dw, rank, world, dist)
        elif rw is not None:
            res = run_softmax(args, rw, rank, world, dist)
        else:
            res = run_ours(args, w, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
