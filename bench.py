"""Benchmark of the single-pass online-softmax attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-e2e]

One step = one fa_fwd call (the whole hot path: QK^T, online softmax, PV,
finalize; for split-KV workloads also the merge) over the workload's inputs.
Default workload: non-causal B=2 H=32 Nq=Nk=4096 d=128, Q x4 (the
configuration the tensor-peak target is quoted on).  Inputs (Q+K+V = 201 MB)
exceed the 129 MB L2 and the L2 is also flushed (a 512 MB write) before every
timed step; the flush is outside the step's CUDA-event pair.

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): replicas only, each
rank runs the same workload on its own GPU; value = sum over ranks of the
work / max over ranks of the time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
row sample of the same workload (there is no other implementation to run).
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
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from online_softmax_sm_gb300 import workloads  # noqa: E402

METRIC = "attention fwd TFLOPS (bf16, 1×GB300) and % of dense BF16 tensor peak"
SOFTMAX_METRIC = "row softmax throughput (two-pass online normaliser), algorithmic GB/s"
FP8_METRIC = "attention fwd TFLOPS (FP8 E4M3 inputs and P, 1×GB300) and % of dense FP8 tensor peak"
BWD_METRIC = "attention bwd TFLOPS (bf16, 1×GB300; 2.5x the forward's FLOPs) and % of dense BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_ALIASES = {"c1": workloads.C1, "c2": workloads.C2, "c3": workloads.C3, "c4": workloads.C4,
                    "c4_masked": workloads.C4_MASKED, "c5": workloads.C5,
                    "local": workloads.LOCAL}
SOFTMAX_ALIASES = {"softmax_f32": workloads.SOFTMAX_F32,
                   "softmax_bf16_vocab": workloads.SOFTMAX_BF16_VOCAB,
                   "softmax_f32_long": workloads.SOFTMAX_F32_LONG}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def workload_of(name: str) -> workloads.Workload:
    """c1..c5 / c4_masked / local, a full workload name, or
    custom:B,H,Nq,Nk,d[,causal[,n_splits[,seed[,window_left,window_right]]]]
    (smaller cases for profiling)."""
    if name in WORKLOAD_ALIASES:
        return WORKLOAD_ALIASES[name]
    if name in workloads.WORKLOADS:
        return workloads.WORKLOADS[name]
    if name.startswith("custom:"):
        f = [int(x) for x in name[len("custom:"):].split(",")]
        B, H, Nq, Nk, d = f[:5]
        causal = bool(f[5]) if len(f) > 5 else False
        n_splits = f[6] if len(f) > 6 else 1
        seed = f[7] if len(f) > 7 else 0
        window = (f[8], f[9]) if len(f) > 9 else None
        return workloads.custom(B, H, Nq, Nk, d, seed=seed, causal=causal, n_splits=n_splits,
                                window=window)
    raise SystemExit(f"unknown workload {name}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


FWD_SOURCES = ["fa_fwd_kernel.cuh", "fa_fwd_d64_bc64.cu", "fa_fwd_d64_bc128.cu",
               "fa_fwd_d128_bc64.cu", "fa_fwd_d128_bc128.cu", "fa_ptx.cuh", "fa_wait.cuh",
               "fa_internal.h"]
SOFTMAX_SOURCES = ["fa_softmax.cu", "fa_ptx.cuh", "fa_wait.cuh", "fa_internal.h"]
BWD_SOURCES = ["fa_bwd_kernel.cuh", "fa_bwd_d64.cu", "fa_bwd_d128.cu", "fa_ptx.cuh", "fa_wait.cuh",
               "fa_internal.h", "fa_status.h"]


def kernel_source_hash(files=None) -> str:
    """Hash of the kernel sources `files` (names under csrc/; all when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "online_softmax_sm_gb300", "csrc")
    names = sorted(files) if files else sorted(os.listdir(csrc))
    for fn in names:
        if fn.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_kernel(workload_name: str, default: str) -> str:
    """Name of the dominant kernel in the committed ncu summary of the
    workload (the kernel its launch list shows), else `default`."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            return json.load(f).get(workload_name, {}).get("kernel", default)
    except (OSError, ValueError):
        return default


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if absent or taken on different kernel sources (the
    entry lists the source files its hash covers)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload_name)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash(ent.get("sources")):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.device_index = device_index
        self.thread = None

    def start(self):
        ident = None
        try:
            props = torch.cuda.get_device_properties(self.device_index)
            ident = "GPU-" + str(props.uuid)
        except Exception:
            ident = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if ident:
            cmd += ["-i", ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first samples arrive before the timed region

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if self.proc is None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = None
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [p for (t, p) in sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]]
            note = "timed region shorter than the 50 ms sampling period; nearest samples"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for nm, val in zip(names, p[5:9]):
                if val.strip().lower() in ("active", "1"):
                    reasons.add(nm)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "reasons": sorted(reasons), "samples": len(inside),
               "power_w_max": max([num(p[3]) for p in inside if num(p[3]) is not None], default=None)}
        if note:
            out["note"] = note
        return out


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(world: int, flops_per_rank: float, ms_local: float, device) -> tuple[float, float]:
    """Replicas: every rank ran the same workload.  Returns (max ms over ranks,
    whole-job TFLOP/s = world * flops / max time)."""
    ms = max_over_ranks(ms_local, world, device)
    return ms, world * flops_per_rank / (ms * 1e-3) / 1e12


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def row_flops(w: workloads.Workload, rows) -> float:
    """Algorithmic FLOPs of the listed query rows: 4*d per visible key."""
    off = w.Nk - w.Nq
    if w.window is not None:
        wl, wr = w.window
        tot = 0
        for r in rows:
            lo = 0 if wl < 0 else max(0, r + off - wl)
            hi = w.Nk - 1 if wr < 0 else min(w.Nk - 1, r + off + wr)
            tot += max(0, hi - lo + 1)
        return 4.0 * w.d * tot
    if not w.causal:
        return 4.0 * w.Nk * w.d * len(rows)
    return float(sum(4.0 * max(0, min(w.Nk, r + off + 1)) * w.d for r in rows))


def oracle_rows(w: workloads.Workload, qh, kh, vh, rows, threads):
    """The oracle on listed rows of one head, with the workload's mask."""
    import oracle

    if w.window is not None:
        return oracle.attention_window(qh, kh, vh, w.scale, w.window[0], w.window[1], rows=rows,
                                       threads=threads)
    return oracle.attention(qh, kh, vh, w.scale, w.causal, rows=rows, threads=threads)


def forward(fa, w: workloads.Workload, q, k, v, o, lse):
    """One call of the library's public forward for this workload's mask
    (o, lse: output buffers, or None to allocate)."""
    if w.window is not None:
        return fa.fwd_local(q, k, v, w.window[0], w.window[1], w.scale, w.n_splits, out=o, lse=lse)
    return fa.fwd(q, k, v, w.scale, w.causal, w.n_splits, out=o, lse=lse, bc=w.bc)


def cpu_oracle_sample(w: workloads.Workload, q, k, v, target_s: float, seed: int = 0,
                      threads: int = 0):
    """Time the oracle on a bounded row sample of the workload (all host
    cores unless `threads` is given); returns a dict."""
    import numpy as np

    import oracle

    threads = threads or oracle.default_threads()
    rng = np.random.default_rng(seed)
    B, H = w.B, w.H
    # per-row cost: 4*Nk_visible*d; calibrate on a small sample first
    head = (0, 0)
    qh, kh, vh = (x[head[0], head[1]].cpu().double().numpy() for x in (q, k, v))

    calib_rows = sorted(rng.choice(w.Nq, size=min(w.Nq, 256), replace=False).tolist())
    t0 = time.perf_counter()
    oracle_rows(w, qh, kh, vh, calib_rows, threads)
    dt = time.perf_counter() - t0
    rate = row_flops(w, calib_rows) / max(dt, 1e-9)
    want_flops = rate * target_s
    total_rows = B * H * w.Nq
    avg_row = w.flops / total_rows
    n_rows = int(min(total_rows, max(256, want_flops / avg_row)))
    # whole heads first, then a partial head
    heads = [(b, h) for b in range(B) for h in range(H)]
    rng.shuffle(heads)
    plan = []
    left = n_rows
    for (b, h) in heads:
        if left <= 0:
            break
        take = min(left, w.Nq)
        rows = None if take == w.Nq else sorted(rng.choice(w.Nq, size=take, replace=False).tolist())
        plan.append(((b, h), rows))
        left -= take
    flops = 0.0
    elapsed = 0.0  # oracle time only (bf16 -> fp64 conversion excluded)
    for (b, h), rows in plan:
        qh, kh, vh = (x[b, h].cpu().double().numpy() for x in (q, k, v))
        rr = rows if rows is not None else list(range(w.Nq))
        ts = time.perf_counter()
        oracle_rows(w, qh, kh, vh, rows, threads)
        elapsed += time.perf_counter() - ts
        flops += row_flops(w, rr)
    return {"tflops": flops / elapsed / 1e12, "seconds": elapsed, "rows": n_rows,
            "heads": len(plan), "threads": threads, "flops": flops}


def run_reference(args, w):
    world, rank, local = dist_setup(args.gpus)
    if rank != 0:
        return
    import numpy as np

    import oracle

    threads = oracle.default_threads()
    q, k, v = workloads.generate(w, device="cpu")
    rng = np.random.default_rng(1)
    per_step_s = min(3.0, 60.0 / max(1, args.steps + args.warmup))  # about a minute in all
    # calibrate rows per step
    qh, kh, vh = (x[0, 0].double().numpy() for x in (q, k, v))
    rows = sorted(rng.choice(w.Nq, size=min(w.Nq, 128), replace=False).tolist())
    t0 = time.perf_counter()
    oracle_rows(w, qh, kh, vh, rows, threads)
    dt = time.perf_counter() - t0
    avg_row = w.flops / (w.B * w.H * w.Nq)
    rows_per_step = int(max(32, min(w.Nq, len(rows) * per_step_s / max(dt, 1e-9))))
    heads_np = {}

    def step(i):
        b = (i // w.H) % w.B
        h = i % w.H
        if (b, h) not in heads_np:
            heads_np[(b, h)] = tuple(x[b, h].double().numpy() for x in (q, k, v))
        qh, kh, vh = heads_np[(b, h)]
        rr = sorted(rng.choice(w.Nq, size=rows_per_step, replace=False).tolist())
        oracle_rows(w, qh, kh, vh, rr, threads)
        return rr

    for i in range(args.warmup):
        step(i)
    times, flops = [], 0.0
    for i in range(args.steps):
        t0 = time.perf_counter()
        rr = step(args.warmup + i)
        times.append(time.perf_counter() - t0)
        flops += row_flops(w, rr)
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{kk: vv for kk, vv in w.describe().items() if kk != "name"}},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} seeded query rows per step, one head per step "
                                   f"(avg {avg_row:.3g} FLOP per row), fp64 three-pass oracle"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import online_softmax_sm_gb300 as fa

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    fa.lib()

    q, k, v = workloads.generate(w, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    launches_per_step = 1 if w.n_splits <= 1 else 2  # split-KV: partials, then the merge

    def step():
        forward(fa, w, q, k, v, o, lse)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fa.device_status(dev) != fa.FA_OK:
        raise SystemExit("device status reports a timed-out wait")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_region0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_region1 = time.time()
    barrier(world)
    sampler.stop()
    if fa.device_status(dev) != fa.FA_OK:
        raise SystemExit("device status reports a timed-out wait")
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_local = statistics.mean(step_ms)
    ms, value = aggregate(world, w.flops, ms_local, dev)

    # ---- dominant kernel: the forward kernel.  Split-KV: the partial kernel
    # (fa_fwd_partial) is timed alone for the kernel's own HBM fraction, and
    # the step (partials + merge, one fa_fwd) gives the step-level fraction.
    peaks, peak_src = load_peaks()
    if w.n_splits > 1 and w.window is None:
        m_p = torch.empty((w.n_splits, w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
        l_p = torch.empty_like(m_p)
        o_p = torch.empty((w.n_splits, w.B, w.H, w.Nq, w.d), dtype=torch.float32, device=dev)
        kt = []
        for i in range(max(10, min(args.steps, 50))):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fa.fwd_partial(q, k, v, w.n_splits, w.scale, w.causal, m_p, l_p, o_p)
            b.record(stream)
            kt.append((a, b))
        torch.cuda.synchronize(dev)
        k_ms = statistics.mean(a.elapsed_time(b) for a, b in kt)
        kern_bytes = (w.B * w.H * w.Nq * w.d + 2 * w.B * w.H * w.Nk * w.d) * 2
        achieved = kern_bytes / (k_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        step_gbs = kern_bytes / (ms_local * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                    "kernel": "fa_fwd_kernel<128,128,1> (split partials)", "kernel_ms": k_ms,
                    "algorithmic_bytes_per_launch": kern_bytes, "peak_source": peak_src + " hbm_gbs",
                    "step_ms": ms_local, "step_achieved": step_gbs, "step_frac": step_gbs / peak}
        del m_p, l_p, o_p
    else:
        achieved = w.flops / (ms_local * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                    "kernel": "fa_fwd_kernel", "kernel_ms": ms_local,
                    "algorithmic_flops_per_launch": w.flops,
                    "peak_source": peak_src + " bf16_tflops (burst: one launch timed alone)"}

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and w.n_splits == 1 and not w.bc:
        # fa_fwd_host (fa_fwd_local_host with a window): the library's host-buffer
        # call (page-locked in/out buffers, copies in, kernels and copies out
        # pipelined over groups of heads); it returns when O and LSE are on the
        # host, so the wall clock times it.
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        n_e2e = max(5, min(args.steps, 30))
        for _ in range(2):
            fa.fwd_host(hq, hk, hv, w.scale, w.causal, out=ho, lse=hl, window=w.window)
        tt = []
        for _ in range(n_e2e):
            t0 = time.perf_counter()
            fa.fwd_host(hq, hk, hv, w.scale, w.causal, out=ho, lse=hl, window=w.window)
            tt.append((time.perf_counter() - t0) * 1e3)
        e_ms = max_over_ranks(statistics.mean(tt), world, dev)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        e2e = {"value": world * w.flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "api": ("fa_fwd_host" if w.window is None else "fa_fwd_local_host")
                      + " (C ABI, host buffers, wall clock)"}
    elif not args.no_e2e:
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        n_e2e = max(5, min(args.steps, 30))

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            forward(fa, w, dq, dk, dv, o, lse)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        tt = []
        for _ in range(n_e2e):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            b.record(stream)
            tt.append((a, b))
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in tt), world, dev)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        e2e = {"value": world * w.flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "api": "pinned torch copies + the device call, one stream, CUDA events"}
        del dq, dk, dv

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = cpu_oracle_sample(w, q, k, v, args.cpu_seconds)
        cpu = {"value": s["tflops"], "unit": "TFLOPS", "cores": s["threads"], "kind": "oracle",
               "sample": f"{s['rows']} seeded query rows over {s['heads']} heads of this workload "
                         f"({s['flops']:.3g} FLOP, {s['seconds']:.1f} s), fp64 three-pass oracle"}
        if w.name in (workloads.C1.name, workloads.C2.name):
            # the two small workloads also get the oracle's single-thread rate
            s1 = cpu_oracle_sample(w, q, k, v, min(args.cpu_seconds, 5.0), threads=1)
            cpu["one_core"] = {"value": s1["tflops"], "unit": "TFLOPS", "cores": 1,
                               "sample": f"{s1['rows']} seeded query rows over {s1['heads']} heads "
                                         f"({s1['flops']:.3g} FLOP, {s1['seconds']:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "causal": w.causal, "n_splits": w.n_splits, "scale": w.scale,
                       "q_mult": w.q_mult, "k_ramp": w.k_ramp, "seed": w.seed,
                       "window": list(w.window) if w.window is not None else None,
                       "l2": "flushed before every timed step (512 MB write); inputs > L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "tensor_peak_frac": value / world / float(peaks["bf16_tflops"])},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": sampler.summary(t_region0, t_region1),
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def softmax_workload_of(name: str):
    """softmax_f32 / softmax_bf16_vocab / softmax_f32_long, a full softmax
    workload name, or softmax:ROWS,COLS,f32|bf16[,seed] (smaller cases)."""
    if name in SOFTMAX_ALIASES:
        return SOFTMAX_ALIASES[name]
    if name.startswith("softmax:"):
        f = name[len("softmax:"):].split(",")
        rows, cols, dt = int(f[0]), int(f[1]), f[2]
        seed = int(f[3]) if len(f) > 3 else 0
        return workloads.SoftmaxWorkload(f"softmax_{dt}_r{rows}c{cols}", rows, cols, dt, seed=seed)
    return workloads.SOFTMAX_WORKLOADS.get(name)


def softmax_oracle_sample(sw, x, target_s: float, seed: int = 0):
    """Time the oracle on seeded rows of x for about target_s seconds."""
    import numpy as np

    import oracle

    threads = oracle.default_threads()
    rng = np.random.default_rng(seed)
    calib = sorted(rng.choice(sw.rows, size=min(sw.rows, 8), replace=False).tolist())
    xs = x[calib].cpu().double().numpy()
    t0 = time.perf_counter()
    oracle.softmax_rows(xs, threads=threads)
    per_row = (time.perf_counter() - t0) / len(calib)
    n = int(min(sw.rows, max(8, target_s / max(per_row, 1e-9))))
    sel = sorted(rng.choice(sw.rows, size=n, replace=False).tolist())
    xs = x[sel].cpu().double().numpy()
    t0 = time.perf_counter()
    oracle.softmax_rows(xs, threads=threads)
    dt = time.perf_counter() - t0
    nbytes = n * (2 * sw.cols * sw.elt + 4)
    return {"gbs": nbytes / dt / 1e9, "seconds": dt, "rows": n, "threads": threads}


def run_softmax(args, sw):
    """The standalone row softmax: one fa_softmax_rows call per step."""
    import online_softmax_sm_gb300 as fa

    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank != 0:
            return
        x = workloads.generate_logits(sw, device="cpu")
        times, nbytes, threads, rows = [], 0, 0, 0
        for i in range(args.warmup + args.steps):
            r = softmax_oracle_sample(sw, x, 2.0, seed=i)
            if i >= args.warmup:
                times.append(r["seconds"])
                nbytes += r["rows"] * (2 * sw.cols * sw.elt + 4)
                threads, rows = r["threads"], r["rows"]
        value = nbytes / sum(times) / 1e9
        line = {"impl": "reference", "metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * sum(times) / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": sw.name, **sw.describe()},
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                 "sample": f"about {rows} seeded rows per step, fp64 two-pass oracle"},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    fa.lib()
    x = workloads.generate_logits(sw, device=dev)
    y = torch.empty_like(x)
    lse = torch.empty(sw.rows, dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step():
        fa.softmax_rows(x, out=y, lse=lse)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_region0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_region1 = time.time()
    barrier(world)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_local = statistics.mean(step_ms)
    ms = max_over_ranks(ms_local, world, dev)
    value = world * sw.io_bytes / (ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    achieved = sw.io_bytes / (ms_local * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": achieved / float(peaks["hbm_gbs"]), "traffic": recorded_traffic(sw.name),
                "kernel": recorded_kernel(sw.name, "fa_softmax_rows"), "kernel_ms": ms_local,
                "algorithmic_bytes_per_launch": sw.io_bytes, "peak_source": peak_src + " hbm_gbs"}

    e2e = None
    if not args.no_e2e:
        hx = x.cpu().pin_memory()
        hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        dx = torch.empty_like(x)

        def e2e_step():
            dx.copy_(hx, non_blocking=True)
            fa.softmax_rows(dx, out=y, lse=lse)
            hy.copy_(y, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        tt = []
        for _ in range(max(5, min(args.steps, 20))):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            b.record(stream)
            tt.append((a, b))
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in tt), world, dev)
        e2e = {"value": world * sw.io_bytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hx.numel() * hx.element_size(),
               "d2h_bytes_per_step": hy.numel() * hy.element_size() + hl.numel() * hl.element_size(),
               "ms_per_step": e_ms}
        del dx

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = softmax_oracle_sample(sw, x, args.cpu_seconds)
        cpu = {"value": r["gbs"], "unit": "GB/s", "cores": r["threads"], "kind": "oracle",
               "sample": f"{r['rows']} seeded rows of this workload ({r['seconds']:.1f} s), "
                         "fp64 two-pass oracle"}
    if rank == 0:
        line = {"metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": sw.dtype, "data": "synthetic",
                "config": {"workload": sw.name, **sw.describe(),
                           "l2": "flushed before every timed step (512 MB write); inputs > L2",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps, "clocks": sampler.summary(t_region0, t_region1),
                "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def oracle_fp8_rows(w: workloads.Workload, q8, k8, v8, b: int, h: int, rows) -> float:
    """The oracle's FP8 forward (Max_offset = 8, descales 1; one host thread)
    on the listed rows of head (b, h).  Returns its wall time in seconds."""
    import oracle

    qh, kh, vh = (x[b, h].float().cpu().double().numpy() for x in (q8, k8, v8))
    t0 = time.perf_counter()
    oracle.attention_fp8(qh, kh, vh, w.scale, 1.0, 1.0, 1.0, w.causal, rows=rows)
    return time.perf_counter() - t0


def fp8_oracle_sample(w: workloads.Workload, q8, k8, v8, target_s: float, seed: int = 0):
    """Time the FP8 oracle on seeded rows of seeded heads for about target_s
    seconds; returns a dict."""
    import numpy as np

    rng = np.random.default_rng(seed)
    calib = sorted(rng.choice(w.Nq, size=min(w.Nq, 16), replace=False).tolist())
    oracle_fp8_rows(w, q8, k8, v8, 0, 0, calib[:1])  # loads the library
    rate = row_flops(w, calib) / max(oracle_fp8_rows(w, q8, k8, v8, 0, 0, calib), 1e-9)
    avg_row = w.flops / (w.B * w.H * w.Nq)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    rng.shuffle(heads)
    flops = elapsed = 0.0
    n_rows = n_heads = 0
    for b, h in heads:
        if elapsed >= target_s:
            break
        take = int(max(8, min(w.Nq, rate * (target_s - elapsed) / avg_row)))
        rows = sorted(rng.choice(w.Nq, size=take, replace=False).tolist())
        elapsed += oracle_fp8_rows(w, q8, k8, v8, b, h, rows)
        flops += row_flops(w, rows)
        n_rows += take
        n_heads += 1
    return {"tflops": flops / elapsed / 1e12, "seconds": elapsed, "rows": n_rows, "heads": n_heads,
            "threads": 1, "flops": flops}


def run_fp8_reference(args, w):
    """--impl reference for the FP8 forward: the oracle's FP8 steps (fp64
    arithmetic, E4M3 rounding of P') on one host thread, each step seeded rows
    of one head (bounded so the whole run takes about a minute)."""
    world, rank, local = dist_setup(args.gpus)
    if rank != 0:
        return
    import numpy as np

    q8, k8, v8 = (t.to(torch.float8_e4m3fn) for t in workloads.generate(w, device="cpu"))
    rng = np.random.default_rng(1)
    per_step_s = min(3.0, 60.0 / max(1, args.steps + args.warmup))
    calib = sorted(rng.choice(w.Nq, size=min(w.Nq, 16), replace=False).tolist())
    oracle_fp8_rows(w, q8, k8, v8, 0, 0, calib[:1])  # loads the library
    rate = row_flops(w, calib) / max(oracle_fp8_rows(w, q8, k8, v8, 0, 0, calib), 1e-9)
    avg_row = w.flops / (w.B * w.H * w.Nq)
    rows_per_step = int(max(8, min(w.Nq, rate * per_step_s / avg_row)))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]

    def step(i):
        b, h = heads[i % len(heads)]
        rows = sorted(rng.choice(w.Nq, size=rows_per_step, replace=False).tolist())
        return oracle_fp8_rows(w, q8, k8, v8, b, h, rows), row_flops(w, rows)

    for i in range(args.warmup):
        step(i)
    total = flops = 0.0
    for i in range(args.steps):
        t, f = step(args.warmup + i)
        total += t
        flops += f
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": FP8_METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + ":fp8", "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": w.causal, "descales": [1.0, 1.0, 1.0]},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} seeded query rows of one head per step, "
                                   f"FP8 oracle (Max_offset = 8) on one thread"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_fp8(args, w):
    """The FP8 forward (fa_fwd_fp8) on the workload's shape: Q, K, V drawn as
    for the bf16 workload and cast to E4M3 (descales 1).  Peak: the measured
    bf16 peak x 2, the nominal FP8 / bf16 ratio of the tensor cores."""
    import online_softmax_sm_gb300 as fa

    if args.impl == "reference":
        return run_fp8_reference(args, w)
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    fa.lib()
    q, k, v = (t.to(torch.float8_e4m3fn) for t in workloads.generate(w, device=dev))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step(qq=q, kk=k, vv=v):
        fa.fwd_fp8(qq, kk, vv, w.scale, 1.0, 1.0, 1.0, w.causal, out=o, lse=lse)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fa.device_status(dev) != fa.FA_OK:
        raise SystemExit("device status reports a timed-out wait")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_region0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_region1 = time.time()
    barrier(world)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_local = statistics.mean(step_ms)
    ms, value = aggregate(world, w.flops, ms_local, dev)
    peaks, peak_src = load_peaks()
    peak = 2.0 * float(peaks["bf16_tflops"])
    achieved = w.flops / (ms_local * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": recorded_traffic(w.name + ":fp8"),
                "kernel": "fa_fwd_kernel<128,128,2,F8>", "kernel_ms": ms_local,
                "algorithmic_flops_per_launch": w.flops,
                "peak_source": peak_src + " bf16_tflops x 2 (nominal FP8 / bf16 dense ratio)"}
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        # fa_fwd_fp8_host: copies in, kernels and copies out pipelined over head
        # groups; it returns with O and LSE on the host, so the wall clock times it
        n_e2e = max(5, min(args.steps, 20))
        for _ in range(2):
            fa.fwd_fp8_host(hq, hk, hv, w.scale, 1.0, 1.0, 1.0, w.causal, out=ho, lse=hl)
        tt = []
        for _ in range(n_e2e):
            t0 = time.perf_counter()
            fa.fwd_fp8_host(hq, hk, hv, w.scale, 1.0, 1.0, 1.0, w.causal, out=ho, lse=hl)
            tt.append((time.perf_counter() - t0) * 1e3)
        e_ms = max_over_ranks(statistics.mean(tt), world, dev)
        e2e = {"value": world * w.flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, hk, hv)),
               "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
               "ms_per_step": e_ms, "api": "fa_fwd_fp8_host (C ABI, host buffers, wall clock)"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s8 = fp8_oracle_sample(w, q, k, v, args.cpu_seconds)
        cpu = {"value": s8["tflops"], "unit": "TFLOPS", "cores": s8["threads"], "kind": "oracle",
               "sample": f"{s8['rows']} seeded query rows over {s8['heads']} heads ({s8['flops']:.3g} "
                         f"FLOP, {s8['seconds']:.1f} s), FP8 oracle (Max_offset = 8) on one thread"}

    if rank == 0:
        line = {"metric": FP8_METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
                "data": "synthetic",
                "config": {"workload": w.name + ":fp8", "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk,
                           "d": w.d, "causal": w.causal, "descales": [1.0, 1.0, 1.0],
                           "l2": "flushed before every timed step (512 MB write); inputs > L2",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps, "clocks": sampler.summary(t_region0, t_region1),
                "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def oracle_bwd_tail(w: workloads.Workload, q, k, v, do, b: int, h: int, nq: int, threads: int) -> float:
    """The oracle's backward for the last nq query rows of head (b, h) with
    every key: under the bottom-right alignment those rows see the same keys
    as in the whole problem.  Returns the oracle's wall time in seconds."""
    import oracle

    tail = slice(w.Nq - nq, w.Nq)
    qh, dh = (x[b, h, tail].detach().cpu().double().numpy() for x in (q, do))
    kh, vh = (x[b, h].detach().cpu().double().numpy() for x in (k, v))
    t0 = time.perf_counter()
    oracle.attention_bwd(qh, kh, vh, dh, w.scale, w.causal, window=w.window, threads=threads)
    return time.perf_counter() - t0


def bwd_tail_flops(w: workloads.Workload, nq: int) -> float:
    """Algorithmic backward FLOPs of the last nq rows: 2.5 x the forward's."""
    return 2.5 * row_flops(w, range(w.Nq - nq, w.Nq))


def bwd_tail_rows(w: workloads.Workload, rate: float, seconds: float) -> int:
    """Rows (from the end) whose backward the oracle runs in about `seconds`
    at `rate` FLOP/s."""
    lo, hi = 16, w.Nq
    while lo < hi:  # the largest tail within the budget (FLOPs grow with the tail)
        mid = (lo + hi + 1) // 2
        if bwd_tail_flops(w, mid) <= rate * seconds:
            lo = mid
        else:
            hi = mid - 1
    return max(16, min(w.Nq, lo))


def bwd_oracle_sample(w: workloads.Workload, q, k, v, do, target_s: float, seed: int = 0):
    """Time the oracle's backward on a bounded sample: the last rows of seeded
    heads, about target_s seconds on all host cores; returns a dict."""
    import numpy as np

    import oracle

    threads = oracle.default_threads()
    rng = np.random.default_rng(seed)
    calib = min(w.Nq, 64)
    oracle_bwd_tail(w, q, k, v, do, 0, 0, 16, threads)  # loads the library
    rate = bwd_tail_flops(w, calib) / max(oracle_bwd_tail(w, q, k, v, do, 0, 0, calib, threads), 1e-9)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    rng.shuffle(heads)
    flops = elapsed = 0.0
    rows = n_heads = 0
    for b, h in heads:
        if elapsed >= target_s:
            break
        nq = bwd_tail_rows(w, rate, target_s - elapsed)
        elapsed += oracle_bwd_tail(w, q, k, v, do, b, h, nq, threads)
        flops += bwd_tail_flops(w, nq)
        rows += nq
        n_heads += 1
    return {"tflops": flops / elapsed / 1e12, "seconds": elapsed, "rows": rows, "heads": n_heads,
            "threads": threads, "flops": flops}


def run_bwd_reference(args, w):
    """--impl reference for the backward: the fp64 oracle's gradients on the
    host cores, each step the last rows of one seeded head (bounded so the
    whole run takes about a minute)."""
    world, rank, local = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle

    threads = oracle.default_threads()
    q, k, v = workloads.generate(w, device="cpu")
    g = torch.Generator().manual_seed(w.seed + 1000)
    do = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    per_step_s = min(3.0, 60.0 / max(1, args.steps + args.warmup))
    calib = min(w.Nq, 64)
    oracle_bwd_tail(w, q, k, v, do, 0, 0, 16, threads)  # loads the library
    rate = bwd_tail_flops(w, calib) / max(oracle_bwd_tail(w, q, k, v, do, 0, 0, calib, threads), 1e-9)
    nq = bwd_tail_rows(w, rate, per_step_s)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    for i in range(args.warmup):
        b, h = heads[i % len(heads)]
        oracle_bwd_tail(w, q, k, v, do, b, h, nq, threads)
    total = 0.0
    for i in range(args.steps):
        b, h = heads[(args.warmup + i) % len(heads)]
        total += oracle_bwd_tail(w, q, k, v, do, b, h, nq, threads)
    flops = bwd_tail_flops(w, nq) * args.steps
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + ":bwd", "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": w.causal, "window": list(w.window) if w.window is not None else None},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"the last {nq} query rows of one head per step with every key "
                                   f"({bwd_tail_flops(w, nq):.3g} FLOP), fp64 oracle gradients"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_bwd(args, w):
    """The attention backward: one fa_bwd call per step (row pass + dK/dV
    kernel + dQ kernel), O, LSE and dO resident.  Algorithmic FLOPs: the five
    products S, dP, dV, dK, dQ = 2.5 x the forward's."""
    import online_softmax_sm_gb300 as fa

    if args.impl == "reference":
        return run_bwd_reference(args, w)
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    fa.lib()
    q, k, v = workloads.generate(w, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 1000)
    do = torch.randn(q.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    o, lse = forward(fa, w, q, k, v, None, None)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    window = w.window if w.window is not None else None
    flops = 2.5 * w.flops

    def step():
        fa.bwd(q, k, v, o, lse, do, w.scale, causal=w.causal, window=window, dq=dq, dk=dk, dv=dv)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fa.device_status(dev) != fa.FA_OK:
        raise SystemExit("device status reports a timed-out wait")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_region0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_region1 = time.time()
    barrier(world)
    sampler.stop()
    if fa.device_status(dev) != fa.FA_OK:
        raise SystemExit("device status reports a timed-out wait")
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_local = statistics.mean(step_ms)
    ms, value = aggregate(world, flops, ms_local, dev)
    peaks, peak_src = load_peaks()
    achieved = flops / (ms_local * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": float(peaks["bf16_tflops"]),
                "unit": "TFLOP/s", "frac": achieved / float(peaks["bf16_tflops"]),
                "traffic": recorded_traffic(w.name + ":bwd"),
                "kernel": "fa_bwd_pre + fa_bwd_dkdv_kernel + fa_bwd_dq_kernel", "kernel_ms": ms_local,
                "algorithmic_flops_per_launch": flops,
                "peak_source": peak_src + " bf16_tflops (burst: one step timed alone)"}
    # ---- end to end: fa_bwd_host (fa_bwd_local_host with a window) on page-locked
    # host buffers: Q, K, V, O, LSE, dO in and dQ, dK, dV out, pipelined over head
    # groups; it returns with the gradients on the host, so the wall clock times it
    e2e = None
    if not args.no_e2e:
        h_in = [x.cpu().pin_memory() for x in (q, k, v, o, lse, do)]
        h_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (dq, dk, dv)]
        n_e2e = max(5, min(args.steps, 20))

        def e2e_step():
            fa.bwd_host(*h_in, w.scale, causal=w.causal, window=window, dq=h_out[0], dk=h_out[1],
                        dv=h_out[2])

        for _ in range(2):
            e2e_step()
        tt = []
        for _ in range(n_e2e):
            t0 = time.perf_counter()
            e2e_step()
            tt.append((time.perf_counter() - t0) * 1e3)
        e_ms = max_over_ranks(statistics.mean(tt), world, dev)
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in h_in),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in h_out),
               "ms_per_step": e_ms,
               "api": ("fa_bwd_host" if window is None else "fa_bwd_local_host")
                      + " (C ABI, host buffers, wall clock)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sb = bwd_oracle_sample(w, q, k, v, do, args.cpu_seconds)
        cpu = {"value": sb["tflops"], "unit": "TFLOPS", "cores": sb["threads"], "kind": "oracle",
               "sample": f"the last rows of {sb['heads']} seeded heads with every key ({sb['rows']} "
                         f"rows, {sb['flops']:.3g} FLOP, {sb['seconds']:.1f} s), fp64 oracle gradients"}

    if rank == 0:
        line = {"metric": BWD_METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": w.name + ":bwd", "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk,
                           "d": w.d, "causal": w.causal,
                           "window": list(w.window) if w.window is not None else None,
                           "l2": "flushed before every timed step (512 MB write); inputs > L2",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": 3 * args.steps, "clocks": sampler.summary(t_region0, t_region1),
                "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.workload.endswith(":bwd"):
        run_bwd(args, workload_of(args.workload[: -len(":bwd")]))
        return
    if args.workload.endswith(":fp8"):
        run_fp8(args, workload_of(args.workload[: -len(":fp8")]))
        return
    sw = softmax_workload_of(args.workload)
    if sw is not None:
        run_softmax(args, sw)
        return
    w = workload_of(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
