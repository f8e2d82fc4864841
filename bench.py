"""Benchmark of the GDN layer on one GB300 (or N independent replicas).

Workload (the pages' "4000-token layer"): chunked prefill of one sequence of
T = 4000 tokens, 16 key / 48 value heads, d_k = d_v = 128, bf16 q/k/v, fp32
g/beta/state, zero initial state.  A step is one prefill call over that
input.  ``value`` is prefill tokens per second per layer, device-timed with
CUDA events, inputs resident in HBM, L2 flushed before every step.  The
decode step (64 sequences x 1 token, 48 heads, fp32 state [64,48,128,128])
is timed in the same run and reported under ``decode`` against HBM bandwidth.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica on its own GPU; the
job value is the tokens of all ranks over the slowest rank's time.
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

METRIC = "GDN prefill tokens/s/layer (T=4000,48 heads) & % bf16 peak; decode % HBM BW"
UNIT = "tokens/s/layer"
PREFILL = dict(seqlens=[4000], Hk=16, Hv=48, d=128)
DECODE = dict(N=64, Hk=16, Hv=48, d=128)
L2_FLUSH_BYTES = 512 << 20          # > 129 MB L2
WORKLOAD = ("GDN prefill, 1 sequence, T=4000, 16 key / 48 value heads, d_k=d_v=128, "
            "bf16 q/k/v, fp32 g/beta/state, zero initial state")
L2_NOTE = "flushed before every step (512 MB write)"
PREFILL_PATHS = ("separate prep and recurrence kernels",
                 "fused: one recurrence per (sequence, value head) beside prep",
                 "fused: one recurrence per value head over all sequences, beside prep")
E2E_PIECES = 4                      # pieces of the end-to-end host-input prefill
# The other two full-size prefill workloads, timed beside the headline one.
EXTRA_PREFILLS = {
    "t20480_initial_state": dict(
        seqlens=[20480], h0=True,
        workload="GDN prefill, 1 sequence, T=20480, 16 key / 48 value heads, d=128, bf16, "
                 "initial state ~N(0,0.02), final state returned"),
    "varlen_8_sequences": dict(
        seqlens=[512, 1000, 2048, 4000, 6000, 8192, 16384, 32768], h0=True,
        workload="GDN varlen prefill, 8 packed sequences {512..32768} (T=70904), 16 key / 48 "
                 "value heads, d=128, bf16, per-sequence initial states, final states returned"),
}


def bench_config(world: int) -> dict:
    """The config dict of both arms' lines (the same workload either way)."""
    return {"workload": WORKLOAD, "l2": L2_NOTE,
            "parallelism": "replicas" if world > 1 else "single GPU"}


def cpu_provenance() -> dict:
    """Host CPU model, the cores this process may run on, and the OpenMP
    threads the oracle uses."""
    import platform

    import oracle
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    affinity = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "affinity_cores": affinity, "omp_threads": oracle.max_threads()}
# Algorithmic work per token per value head (d = 128, C = 64, G = 3), the
# triangle-aware chunked count: 6 d^2 + C (dk + dv) + C dv + 2 C dk / G + C^2 / 3.
FLOPS_PER_TOKEN_HEAD = 6 * 128 ** 2 + 64 * 256 + 64 * 128 + 2 * 64 * 128 // 3 + 64 ** 2 // 3
# Its split between the two main kernels: the recurrence (state products
# 6 d^2, U^T and Delta^T P^T 2 C d_v) and prep (W C d_k, K K^T and Q K^T
# 2 C d_k / G, the triangular inverse C^2 / 3).
FLOPS_RECURRENCE = 6 * 128 ** 2 + 2 * 64 * 128
FLOPS_PREP = FLOPS_PER_TOKEN_HEAD - FLOPS_RECURRENCE
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def flops_of(T, Hv):
    """Algorithmic flops of a prefill of T tokens over Hv value heads."""
    return T * Hv * FLOPS_PER_TOKEN_HEAD


def code_digest(path):
    """SHA-256 of a source file's code: `//` comments, surrounding blanks and
    empty lines dropped, so that a comment edit keeps a recorded profile valid
    and any code change voids it."""
    import hashlib
    lines = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            code = line.split("//", 1)[0].strip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def recorded_traffic(kernel):
    """DRAM bytes per launch (read + write) of `kernel` from the committed ncu
    summary, or None when the kernel's code has changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "prefill_traffic.json")) as f:
            rec = json.load(f)
        digest = code_digest(os.path.join(ROOT, "gated_deltanet_linear_chunk_gb300", "csrc",
                                          "prefill_tc.cu"))
    except (OSError, ValueError):
        return None
    if rec.get("code_sha256") != digest or kernel not in rec.get("bytes_per_launch", {}):
        return None
    return rec["bytes_per_launch"][kernel]


def prefill_bytes(T, Hk, Hv, d):
    """Compulsory HBM bytes of one prefill: q, k, v read, out written (bf16),
    g and beta read (fp32)."""
    return T * (2 * Hk * d * 2 + Hv * d * 2 + Hv * d * 2 + 2 * Hv * 4)


def verify_bytes(N, K, Hk, Hv, d, state_bytes):
    """Compulsory HBM bytes of one verify call: the state read once, K state
    slots written, K tokens of q/k/v read and out written (bf16), g and beta."""
    return N * (Hv * d * d * state_bytes * (1 + K) +
                K * (2 * Hk * d * 2 + 2 * Hv * d * 2 + 2 * Hv * 4))


def verify_inputs(N, K, Hk, Hv, d):
    """K consecutive decode-step inputs per sequence, stacked [N, K, ...]."""
    import torch
    from gated_deltanet_linear_chunk_gb300 import inputs
    xs = [inputs.decode_step_inputs(j, N, Hk, Hv, d, d) for j in range(K)]
    return [torch.stack([getattr(x, f) for x in xs], dim=1).contiguous()
            for f in ("q", "k", "v", "g", "beta")]


def decode_bytes(N, Hk, Hv, d, state_bytes=4):
    """Compulsory HBM bytes of one decode step: the state read and written
    (fp32, or 2 bytes per element when stored in 16 bits), q/k/v read and out
    written (bf16), g and beta read (fp32)."""
    return N * (2 * Hv * d * d * state_bytes + 2 * Hk * d * 2 + 2 * Hv * d * 2 + 2 * Hv * 4)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units of every rank over the slowest rank."""
    return units_per_rank * world / max_seconds


def oracle_sample_prefill(tokens: int, num_threads: int = 0, min_seconds: float = 0.0):
    """Times the fp64 oracle on the first ``tokens`` tokens of the prefill
    workload, all 48 value heads, repeated until ``min_seconds`` have passed
    (at least once).  Returns (tokens/s/layer, seconds, threads, repeats)."""
    import torch

    import oracle
    from gated_deltanet_linear_chunk_gb300 import inputs
    p = inputs.prefill_inputs([tokens], PREFILL["Hk"], PREFILL["Hv"], PREFILL["d"],
                              PREFILL["d"], dtype=torch.bfloat16, seed=0)
    arrs = [x.double().numpy() for x in (p.q, p.k, p.v, p.g, p.beta)]
    threads = num_threads or oracle.max_threads()
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.prefill(*arrs, p.cu_seqlens.numpy(), None, num_threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or reps >= 200:
            break
    # One OpenMP task per (sequence, value head): at most Hv threads work.
    return tokens * reps / dt, dt, min(threads, PREFILL["Hv"]), reps


def run_reference(args, rank):
    """The oracle as the reference arm: fp64 CPU, bounded sample per step."""
    if rank != 0:
        return
    tokens = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample_prefill(max(16, tokens // 8))[0]
    vals, secs = [], []
    threads = 1
    for _ in range(args.steps):
        v, s, threads, _ = oracle_sample_prefill(tokens)
        vals.append(v)
        secs.append(s)
    value = statistics.median(vals)
    sample = (f"first {tokens} of the 4000 tokens, all 48 value heads, fp64 token "
              f"recurrence; tokens/s/layer = tokens / wall time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample, "sample_tokens": tokens,
                         "timing": f"median over {args.steps} steps", **cpu_provenance()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch

    import gated_deltanet_linear_chunk_gb300 as gdn
    from gated_deltanet_linear_chunk_gb300 import inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdn.library()
    gdn.gdn_prefill_fused_mode(args.fused_mode)
    peaks, peak_kind = load_peaks()
    stream = torch.cuda.current_stream()

    # ---------------- prefill ----------------
    P = PREFILL
    p = inputs.prefill_inputs(P["seqlens"], P["Hk"], P["Hv"], P["d"], P["d"],
                              dtype=torch.bfloat16, seed=0)
    T = sum(P["seqlens"])
    dq, dk_, dv = p.q.to(dev), p.k.to(dev), p.v.to(dev)
    dg, db, dcu = p.g.to(dev), p.beta.to(dev), p.cu_seqlens.to(dev)
    out = torch.empty((T, P["Hv"], P["d"]), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def prefill():
        gdn.gdn_chunk_prefill(dq, dk_, dv, dg, db, dcu, None, out=out)

    for _ in range(max(3, args.warmup)):
        prefill()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            prefill()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier()
        # Per-kernel times: the same steps again through the timed entry
        # point, which records events between its launches on this stream
        # (kept out of the headline steps: the launches then go without
        # programmatic dependent launch and the records cost a few us).
        kernel_ms, fused = [], []
        tev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            _, _, f, _ = gdn.gdn_chunk_prefill_timed(dq, dk_, dv, dg, db, dcu, None, out=out,
                                                     events=tev[i])
            fused.append(f)
        torch.cuda.synchronize()
        kernel_ms = [[ev[j].elapsed_time(ev[j + 1]) for j in range(3)] for ev in tev]
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = statistics.median(step_ms)
    ms = max_over_ranks(ms_local, dev)
    value = job_throughput(T, world, ms / 1e3)
    launches_per_step = gdn.prefill_launches(P["Hv"], P["d"], torch.bfloat16)

    flops = T * P["Hv"] * FLOPS_PER_TOKEN_HEAD
    peak_tf = peaks["bf16_tflops"]
    # Roofline of the dominant kernel: its algorithmic flops per launch over
    # its mean launch time in the timed steps.
    # (When the call runs prep and the recurrence as one fused launch, that
    # launch is the kernel, with the whole call's algorithmic flops.)
    ran_fused = all(fused)
    if ran_fused:
        launches_per_step = 2  # chunk table + the fused kernel
    names = ("chunk_table", "prep", "fused") if ran_fused else ("chunk_table", "prep", "recurrence")
    k_us = {name: 1e3 * statistics.mean(m[i] for m in kernel_ms) for i, name in enumerate(names)}
    if ran_fused:
        del k_us["prep"]
        k_flops = {"fused": flops_of(T, P["Hv"])}
    else:
        k_flops = {"recurrence": T * P["Hv"] * FLOPS_RECURRENCE, "prep": T * P["Hv"] * FLOPS_PREP}
    per_kernel = {n: {"us": k_us[n], "flops_per_launch": k_flops[n],
                      "achieved": k_flops[n] / (k_us[n] / 1e6) / 1e12,
                      "frac": k_flops[n] / (k_us[n] / 1e6) / 1e12 / peak_tf,
                      "traffic": recorded_traffic(n)} for n in k_flops}
    # The longer kernel; within 2 % (a tie: their event times differ by less
    # than the timer's resolution) the recurrence, which holds 88 % of the
    # algorithmic work.
    if ran_fused:
        dom = "fused"
    else:
        dom = "prep" if k_us["prep"] > 1.02 * k_us["recurrence"] else "recurrence"
    dom_flops = k_flops[dom]
    achieved_tf = per_kernel[dom]["achieved"]
    traffic = per_kernel[dom]["traffic"]
    pbytes = prefill_bytes(T, P["Hk"], P["Hv"], P["d"])

    # ---------------- the same call writing chunk-boundary snapshots ---------
    snap_res = {}
    for stride in (8, 1):
        snaps = torch.empty((gdn.gdn_chunk_prefill_snapshot_slots(1, T, P["Hk"], P["Hv"], P["d"],
                                                                  P["d"], stride),
                             P["Hv"], P["d"], P["d"]), dtype=torch.float32, device=dev)
        for _ in range(3):
            gdn.gdn_chunk_prefill_snapshots(dq, dk_, dv, dg, db, dcu, None, out=out,
                                            snapshots=snaps, snapshot_chunks=stride)
        snap_ms = []
        for _ in range(5):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gdn.gdn_chunk_prefill_snapshots(dq, dk_, dv, dg, db, dcu, None, out=out,
                                            snapshots=snaps, snapshot_chunks=stride)
            e1.record(stream)
            torch.cuda.synchronize()
            snap_ms.append(e0.elapsed_time(e1))
        nsnap = -(-((T + 63) // 64) // stride)
        snap_res[f"every_{stride}_chunks"] = {
            "us_per_call": 1e3 * statistics.median(snap_ms), "snapshots": nsnap,
            "snapshot_bytes": nsnap * P["Hv"] * P["d"] * P["d"] * 4}
        del snaps

    # ---------------- chunk-parallel scan against the sequential chain -------
    def median_us(fn, n=5):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return 1e3 * statistics.median(ts)

    scan_res = {}
    for sHk, sHv in ((4, 12), (16, 48)):
        ps = inputs.prefill_inputs([20480], sHk, sHv, P["d"], P["d"], dtype=torch.bfloat16, seed=0)
        sa = [x.to(dev) for x in (ps.q, ps.k, ps.v, ps.g, ps.beta, ps.cu_seqlens)]
        sout = torch.empty((20480, sHv, P["d"]), dtype=torch.bfloat16, device=dev)
        seq_us = median_us(lambda: gdn.gdn_chunk_prefill(*sa, out=sout))
        scan_us = median_us(lambda: gdn.gdn_chunk_prefill_scan(*sa, out=sout, chunks_per_group=0))
        scan_res[f"heads_{sHk}_{sHv}"] = {
            "workload": f"1 sequence, T=20480 (320 chunks), {sHk} key / {sHv} value heads, d=128",
            "sequential_us": seq_us, "scan_us": scan_us, "speedup": seq_us / scan_us,
            "tokens_per_s_scan": 20480 / (scan_us / 1e6)}
        del ps, sa, sout
    gdn._workspaces.clear()

    # ---------------- the other full-size prefill workloads ----------------
    extra = {}
    for name, cfg in EXTRA_PREFILLS.items():
        px = inputs.prefill_inputs_on_device(cfg["seqlens"], P["Hk"], P["Hv"], P["d"], P["d"],
                                             dev, seed=0,
                                             initial_state_std=0.02 if cfg["h0"] else None)
        Tx = sum(cfg["seqlens"])
        xout = torch.empty((Tx, P["Hv"], P["d"]), dtype=torch.bfloat16, device=dev)
        xfin = torch.empty_like(px.initial_state) if px.initial_state is not None else None
        xargs = (px.q, px.k, px.v, px.g, px.beta, px.cu_seqlens, px.initial_state)
        x_us = median_us(lambda: gdn.gdn_chunk_prefill(*xargs, out=xout, final_state=xfin),
                         n=10)
        # which kernels the call runs (the timed entry point reports it)
        _, _, xf, _ = gdn.gdn_chunk_prefill_timed(*xargs, out=xout, final_state=xfin)
        torch.cuda.synchronize()
        xflops = flops_of(Tx, P["Hv"])
        extra[name] = {"workload": cfg["workload"], "us_per_call": x_us,
                       "path": PREFILL_PATHS[int(xf)],
                       "tokens_per_s_per_layer": Tx / (x_us / 1e6),
                       "tflops": xflops / (x_us / 1e6) / 1e12,
                       "frac_of_bf16_peak": xflops / (x_us / 1e6) / 1e12 / peak_tf,
                       "flops_per_call": xflops,
                       "inputs": "drawn on the device (torch generator, same recipe)"}
        del px, xout, xfin, xargs
    gdn._workspaces.clear()

    # ---------------- end to end through host buffers ----------------
    hq, hk, hv = (x.pin_memory() for x in (p.q, p.k, p.v))
    hg, hb, hcu = (x.pin_memory() for x in (p.g, p.beta, p.cu_seqlens))
    hout = torch.empty_like(out, device="cpu").pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hg, hb, hcu))
    d2h = hout.numel() * hout.element_size()

    def e2e_serial():
        for dst, src in ((dq, hq), (dk_, hk), (dv, hv), (dg, hg), (db, hb), (dcu, hcu)):
            dst.copy_(src, non_blocking=True)
        prefill()
        hout.copy_(out, non_blocking=True)

    def e2e_pipelined():
        # The public host-input entry point: the sequence in pieces, uploads,
        # computation and downloads overlapped.
        gdn.gdn_chunk_prefill_host(hq, hk, hv, hg, hb, hout, pieces=E2E_PIECES)

    def e2e_time(step):
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            e_s[i].record(stream)
            step()
            e_e[i].record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in zip(e_s, e_e)), dev)

    e2e_ms = e2e_time(e2e_pipelined)
    e2e_serial_ms = e2e_time(e2e_serial)
    h2d -= hcu.numel() * hcu.element_size()  # the pipelined call takes no cu_seqlens

    # ---------------- decode ----------------
    D = DECODE
    state = inputs.decode_state(D["N"], D["Hv"], D["d"], D["d"]).to(dev)
    dsteps = [inputs.decode_step_inputs(s, D["N"], D["Hk"], D["Hv"], D["d"], D["d"])
              for s in range(args.decode_steps)]
    dsteps = [[t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta)] for x in dsteps]
    dout = torch.empty((D["N"], D["Hv"], D["d"]), dtype=torch.bfloat16, device=dev)
    for s in range(3):
        x = dsteps[s % len(dsteps)]
        gdn.gdn_decode_step(*x, state, out=dout)
    torch.cuda.synchronize()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    barrier()
    d0.record(stream)
    for s in range(args.decode_steps):
        gdn.gdn_decode_step(*dsteps[s], state, out=dout)
    d1.record(stream)
    torch.cuda.synchronize()
    dec_us = 1e3 * d0.elapsed_time(d1) / args.decode_steps
    dbytes = decode_bytes(D["N"], D["Hk"], D["Hv"], D["d"])
    dec_gbs = dbytes / (dec_us / 1e6) / 1e9
    # The same steps with the state stored in fp16 (the pages' fork).  One
    # fp16 state (101 MB) fits in L2, so successive steps alternate between
    # two independent batches' states (201 MB together, larger than L2).
    state16 = [inputs.decode_state(D["N"], D["Hv"], D["d"], D["d"]).to(torch.float16).to(dev)
               for _ in range(2)]
    del state
    for s in range(3):
        gdn.gdn_decode_step_half_state(*dsteps[s % len(dsteps)], state16[s % 2], out=dout)
    torch.cuda.synchronize()
    barrier()
    d0.record(stream)
    for s in range(args.decode_steps):
        gdn.gdn_decode_step_half_state(*dsteps[s], state16[s % 2], out=dout)
    d1.record(stream)
    torch.cuda.synchronize()
    dec16_us = 1e3 * d0.elapsed_time(d1) / args.decode_steps
    dbytes16 = decode_bytes(D["N"], D["Hk"], D["Hv"], D["d"], state_bytes=2)
    dec16_gbs = dbytes16 / (dec16_us / 1e6) / 1e9
    del state16

    # ---------------- verify step (8 tokens per sequence, a slot per token) --------
    K = 8
    vx = [t.to(dev) for t in verify_inputs(D["N"], K, D["Hk"], D["Hv"], D["d"])]
    vout = torch.empty((D["N"], K, D["Hv"], D["d"]), dtype=torch.bfloat16, device=dev)
    verify = {}
    for name, sdt, sb in (("fp32_state", torch.float32, 4), ("fp16_state", torch.float16, 2)):
        vstate = inputs.decode_state(D["N"], D["Hv"], D["d"], D["d"]).to(sdt).to(dev)
        vslots = torch.empty((D["N"], K, D["Hv"], D["d"], D["d"]), dtype=sdt, device=dev)
        for _ in range(3):
            gdn.gdn_verify_step(*vx, vstate, slots=vslots, out=vout)
        torch.cuda.synchronize()
        barrier()
        reps = 20
        d0.record(stream)
        for _ in range(reps):
            gdn.gdn_verify_step(*vx, vstate, slots=vslots, out=vout)
        d1.record(stream)
        torch.cuda.synchronize()
        v_us = 1e3 * d0.elapsed_time(d1) / reps
        vbytes = verify_bytes(D["N"], K, D["Hk"], D["Hv"], D["d"], sb)
        verify[name] = {"us_per_call": v_us, "tokens_per_s": D["N"] * K / (v_us / 1e6),
                        "bytes_per_call": vbytes, "achieved_gbs": vbytes / (v_us / 1e6) / 1e9,
                        "frac": vbytes / (v_us / 1e6) / 1e9 / peaks["hbm_gbs"]}
        del vstate, vslots

    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world),
        "timing": {"ms_per_step": "median of the timed steps", "mean_ms": statistics.mean(step_ms),
                   "min_ms": min(step_ms), "max_ms": max(step_ms)},
        "gpu_launches": launches_per_step * args.steps,
        "prefill_fused_mode": args.fused_mode,
        "roofline": {"bound": "tensor", "achieved": achieved_tf, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": achieved_tf / peak_tf, "traffic": traffic,
                     "kernel": dom, "kernel_us": k_us[dom],
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "flops_per_launch": dom_flops, "per_kernel": per_kernel,
                     "whole_prefill": {"flops": flops, "tflops": flops / (ms_local / 1e3) / 1e12,
                                       "frac": flops / (ms_local / 1e3) / 1e12 / peak_tf,
                                       "algorithmic_bytes": pbytes}},
        "kernels_us": {n: {"us": v, "share": v / sum(k_us.values())} for n, v in k_us.items()},
        "e2e": {"value": job_throughput(T, world, e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": f"gdn_chunk_prefill_host (pinned host buffers, {E2E_PIECES} pieces)",
                "serial_copies": {"value": job_throughput(T, world, e2e_serial_ms / 1e3),
                                  "note": "copies, gdn_chunk_prefill and the read-back "
                                          "one after another on one stream"}},
        "decode": {"workload": "64 sequences x 1 token, 16 key / 48 value heads, d=128, "
                               "fp32 state, bf16 q/k/v",
                   "us_per_step": dec_us, "steps": args.decode_steps,
                   "bytes_per_step": dbytes, "achieved_gbs": dec_gbs,
                   "peak_gbs": peaks["hbm_gbs"], "frac": dec_gbs / peaks["hbm_gbs"],
                   "frac_of_8tbs": dec_gbs / 8000.0, "peak_kind": peak_kind},
        "decode_f16_state": {"workload": "as decode, state stored in fp16 (fp32 math); "
                                         "steps alternate between two such batches' states "
                                         "so that the 101 MB state is not served from L2",
                             "us_per_step": dec16_us, "steps": args.decode_steps,
                             "bytes_per_step": dbytes16, "achieved_gbs": dec16_gbs,
                             "peak_gbs": peaks["hbm_gbs"], "frac": dec16_gbs / peaks["hbm_gbs"],
                             "speedup_vs_fp32_state": dec_us / dec16_us},
        "prefill_other_workloads": extra,
        "prefill_with_snapshots": snap_res,
        "prefill_scan": scan_res,
        "verify": {"workload": "64 sequences x 8 tokens from one state, a state slot per "
                               "token, 16/48 heads, d=128, bf16 q/k/v", **verify},
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rank == 0 and not args.no_cpu_baseline:
        v, s, threads, reps = oracle_sample_prefill(args.ref_tokens, min_seconds=10.0)
        line["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {args.ref_tokens} of the 4000 tokens, all 48 value heads, "
                      f"{reps} repeats (fp64 token recurrence, {s:.1f} s wall)",
            **cpu_provenance()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_case(args):
    """--prefill-case: one packed prefill batch alone (16 key / 48 value heads,
    d = 128, bf16, initial states, the bench's input recipe drawn on the
    device), `warmup` calls then `steps` timed calls with the L2 flushed before
    each.  For profiling a prefill path on a case small enough to capture;
    prints one JSON line (not the bench's result line)."""
    import torch
    import gated_deltanet_linear_chunk_gb300 as gdn
    from gated_deltanet_linear_chunk_gb300 import inputs
    dev = torch.device("cuda")
    lens = [int(x) for x in args.prefill_case.split(",")]
    gdn.gdn_prefill_fused_mode(args.fused_mode)
    P = PREFILL
    p = inputs.prefill_inputs_on_device(lens, P["Hk"], P["Hv"], P["d"], P["d"], dev, seed=0,
                                        initial_state_std=0.02)
    T = sum(lens)
    out = torch.empty((T, P["Hv"], P["d"]), dtype=torch.bfloat16, device=dev)
    fin = torch.empty_like(p.initial_state)
    xargs = (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens, p.initial_state)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        gdn.gdn_chunk_prefill(*xargs, out=out, final_state=fin)
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gdn.gdn_chunk_prefill(*xargs, out=out, final_state=fin)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    _, _, f, _ = gdn.gdn_chunk_prefill_timed(*xargs, out=out, final_state=fin)
    torch.cuda.synchronize()
    us = statistics.median(ts)
    print(json.dumps({"prefill_case": lens, "tokens": T, "us_per_call": us,
                      "tokens_per_s_per_layer": T / (us / 1e6), "path": PREFILL_PATHS[int(f)],
                      "steps": args.steps, "warmup": args.warmup}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--ref-tokens", type=int, default=4000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-mode", type=int, choices=(0, 1, 2, 3), default=2,
                    help="when the prefill uses its fused prep + recurrence kernel "
                         "(gdn_prefill_fused_mode: 0 never, 1 whenever it fits, "
                         "2 by the library's cost model, its default, 3 the variant with "
                         "one recurrence per value head whenever it fits)")
    ap.add_argument("--prefill-case", default=None, metavar="LENS",
                    help="time one packed prefill batch alone (comma-separated sequence "
                         "lengths, 16/48 heads) instead of the bench, for profiling")
    args = ap.parse_args(argv)
    if args.prefill_case:
        run_case(args)
        return
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, world, local)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
