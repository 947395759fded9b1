#!/usr/bin/env python3
"""Throughput of the ReplaySSM decode path on GB300.

Workload: one Mamba-2-shaped SSM layer. B=256 sequences, H=128 value heads,
P=64, N=128 (a 4 MiB FP32 checkpoint per sequence), G=8 groups, window L=16,
bf16 v/k/q. One bench step is one full window of L decode launches over the
batch: L-1 non-flush steps plus the flush step. The metric is seq-steps/s,
that is, (sequence, decode step) pairs per second.

Prints one JSON line. Keys beyond the driver contract:
  roofline      achieved HBM GB/s of the decode kernel (algorithmic bytes per
                launch / mean launch time from CUDA events on its stream)
                against the measured copy bandwidth
  cpu_baseline  the float64 CPU oracle on a bounded sample of the same workload
  e2e           the same metric with inputs copied from pinned host memory and
                outputs copied back inside the timed region
  comparison    the conventional read-update-write kernel on the same workload
  verify_b512_t4, delta_verify_b512_t4, read_copy_e4m3, read_copy_e2m1, delta_rule,
  ckpt_f16_sr, ckpt_f16_rn
                the secondary arms of the path, each with its own roofline
                block: speculative rounds (verify + commit + flush, B=512,
                T=4) against the snapshot comparator, the same rounds of a
                gated delta-rule layer, decode windows reading
                an E4M3 or E2M1 copy of the checkpoint, decode windows of
                a gated delta-rule layer of the same shape, and decode windows
                with the checkpoint stored as binary16 (stochastic rounding,
                or rounding to nearest)
  static_scratch
                the headline windows through the entry point that keeps its
                tickets in a static device array, timed in alternating blocks
                with the ordinary decode step on one layer

The timed region covers at least --min-seconds of windows (default 1 s), and
at least --steps of them, so that the clock sampler sees several samples.
`--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SSM decode seq-steps/s at B=256, L=16; achieved HBM GB/s vs GB300 peak"
UNIT = "seq-steps/s"
WORKLOAD = synth.PRESETS["mamba2_layer_b256_l16"]
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes per launch from ncu captures, keyed by workload, each with the hash
# of the kernel sources it was taken on (written beside the summaries).
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


# ----------------------------------------------------------------- analytic bytes
def record_bytes(s, delta: bool = False) -> int:
    """Bytes of one input record (alpha, v, k; and beta for a delta-rule layer) of one sequence."""
    es = 2 if s.in_dtype == "bf16" else 4
    return 4 * s.H * (2 if delta else 1) + es * s.H * s.P + es * s.G * s.N


def copy_bytes_per_head(s, read_fmt) -> int:
    """Bytes of one head's read copy (codes + scales, padded to 16)."""
    if read_fmt is None:
        return 0
    P, N = s.P, s.N
    if read_fmt == "e4m3":
        return -(-(P * N + 4 * P) // 16) * 16
    rsc = -(-(P * N // 2 + P * N // 16) // 16) * 16
    return -(-(rsc + 4 * P) // 16) * 16


def window_bytes(s, read_fmt=None, ckpt_bytes: int = 4, delta: bool = False) -> dict:
    """Algorithmic HBM bytes of one sequence over one window of L decode steps.

    Every step reads its inputs (record + q) and writes its output. Step t of
    the window (t = 0..L-1) also reads the t buffered records, and every
    non-flush step appends its record. The L-1 non-flush steps each read the
    checkpoint |S|, or its read copy |C| when there is one. The flush step
    reads |S| and writes it once, plus the refreshed copy. ckpt_bytes is the
    checkpoint's element size (2 for an FP16 checkpoint). A delta-rule layer's
    inputs carry beta too, and its buffered records hold the fp32 pseudo-value
    w in place of v.
    """
    es = 2 if s.in_dtype == "bf16" else 4
    S = ckpt_bytes * s.H * s.P * s.N
    C = s.H * copy_bytes_per_head(s, read_fmt)
    ring_rec = 4 * s.H + (4 if delta else es) * s.H * s.P + es * s.G * s.N  # a buffered record
    inp = record_bytes(s, delta) + es * s.G * s.N                            # a step's inputs
    out = 4 * s.H * s.P
    L = s.L
    reads = (L - 1) * (C if read_fmt else S) + S
    total = reads + S + C + ring_rec * L * (L - 1) // 2 + L * (inp + out) + (L - 1) * ring_rec
    conv = L * (2 * 4 * s.H * s.P * s.N + inp + out)
    # per launch: a non-flush step at window position t reads t buffered records and
    # appends one (averaged over t = 0..L-2); the flush step reads L-1 records
    nonflush = (C if read_fmt else S) + ring_rec * (L - 2) / 2 + inp + out + ring_rec if L > 1 else 0.0
    flush = 2 * S + C + ring_rec * (L - 1) + inp + out
    return {"replay_window": total, "replay_per_seq_step": total / L, "conventional_per_seq_step": conv / L,
            "state": S, "nonflush_per_seq_launch": nonflush, "flush_per_seq_launch": flush}


# ----------------------------------------------------------------- environment
def measured_peak_gbs() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(sources) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(key: str) -> float | None:
    """DRAM bytes per launch of a workload from profiles/traffic.json, while the kernel
    sources still hash to the value recorded with the capture; else None."""
    try:
        with open(TRAFFIC_JSON) as f:
            entry = json.load(f)[key]
        if entry["kernel_source_sha256"] != kernel_source_hash(entry["kernel_sources"]):
            return None
        return float(entry["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region
    (off with --no-clocks, e.g. under a profiler, which would attach to the sampler)."""

    enabled = True

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        if not ClockSampler.enabled:
            return self
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict | None:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (every rank gets it)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle timing
MAX_ORACLE_THREADS = 64  # bounds the sample's host memory (about 160 MB per thread of 4 sequences)


def usable_cores() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def host_cores() -> int:
    """Threads for the CPU oracle sample: the usable cores, at most MAX_ORACLE_THREADS."""
    return max(1, min(usable_cores(), MAX_ORACLE_THREADS))


class OracleSample:
    """The float64 oracle's recurrence (its definition, as it stands) on a sample of
    the workload: `threads` disjoint groups of `n_seq` sequences, each group with
    its own seeded state and inputs, stepped by one host thread. numpy releases
    the GIL inside its array loops, so the groups run on separate cores."""

    def __init__(self, shape, n_seq: int, threads: int, delta: bool = False, seed: int = 0):
        import oracle
        self.step = oracle.delta_step if delta else oracle.conventional_step
        self.n_seq, self.threads = n_seq, threads
        draw = synth.delta_step_inputs if delta else synth.decode_step_inputs
        s = shape.with_(B=n_seq)
        self.parts = []
        for t in range(threads):
            gen = synth.make_generator(seed + 7919 * t)
            S = oracle.to_f64(synth.initial_state(s, gen))
            self.parts.append([S, [tuple(oracle.to_f64(x) for x in draw(s, gen)) for _ in range(4)]])
        self.done = 0  # steps already taken by every group

    def run(self, n_steps: int) -> float:
        """Wall seconds for n_steps more steps of every group, the threads started together."""
        start = threading.Barrier(self.threads + 1)
        errors = []

        def work(part):
            start.wait()
            try:
                S, steps = part
                for i in range(self.done, self.done + n_steps):
                    S, _ = self.step(S, *steps[i % len(steps)])
                part[0] = S
            except Exception as e:  # surfaced below
                errors.append(e)

        ths = [threading.Thread(target=work, args=(p,)) for p in self.parts]
        for th in ths:
            th.start()
        start.wait()
        t0 = time.perf_counter()
        for th in ths:
            th.join()
        t = time.perf_counter() - t0
        if errors:
            raise errors[0]
        self.done += n_steps
        return t

    def units(self, n_steps: int) -> int:
        return self.threads * self.n_seq * n_steps


def cpu_baseline_line(shape, budget_s: float = 12.0, delta: bool = False) -> dict:
    n_seq, threads = 4, host_cores()
    sample = OracleSample(shape, n_seq, threads, delta=delta)
    sample.run(1)  # first touch of every group's arrays
    per_step = sample.run(2) / 2
    steps = max(4, int(budget_s / max(per_step, 1e-6)))
    t = sample.run(steps)
    what = "gated delta rule" if delta else "conventional recurrence"
    return {"value": sample.units(steps) / t, "unit": UNIT, "cores": usable_cores(), "threads": threads,
            "kind": "oracle",
            "sample": f"float64 {what}, {threads} threads x {n_seq} sequences (of {shape.B}) x all {shape.H} "
                      f"heads, {steps} steps ({t:.1f} s); numpy elementwise, one thread per sequence group"}


# ----------------------------------------------------------------- GPU arm
def decode_pool(s, ls, dev, gen, delta: bool, n: int = 16):
    """n resident steps of seeded inputs (alpha, v, k, q[, beta]) on the device."""
    pool = []
    sc = 1.0 / math.sqrt(s.N)
    for _ in range(n):
        u = torch.randn((s.B, s.H), generator=gen, device=dev)
        alpha = torch.exp(-torch.nn.functional.softplus(u)).float()
        v = (torch.randn((s.B, s.H, s.P), generator=gen, device=dev) * sc).to(ls.torch_in_dtype)
        k = (torch.randn((s.B, s.G, s.N), generator=gen, device=dev) * sc).to(ls.torch_in_dtype)
        q = (torch.randn((s.B, s.G, s.N), generator=gen, device=dev) * sc).to(ls.torch_in_dtype)
        if delta:  # write strengths in (0, 1); unit-norm keys and queries
            beta = torch.sigmoid(torch.randn((s.B, s.H), generator=gen, device=dev)).float()
            k = (k.float() / k.float().norm(dim=-1, keepdim=True)).to(ls.torch_in_dtype)
            q = (q.float() / q.float().norm(dim=-1, keepdim=True)).to(ls.torch_in_dtype)
            pool.append((alpha, v, k, q, beta))
        else:
            pool.append((alpha, v, k, q))
    return pool


class DecodeArm:
    """Decode windows of one layer: the model, its resident inputs and the timing loops."""

    def __init__(self, s, local: int, rank: int, read_fmt=None, ckpt: str = "f32", recurrence: str = "outer"):
        from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM

        self.s, self.read_fmt, self.ckpt_fmt = s, read_fmt, ckpt
        self.delta = recurrence == "delta"
        self.ls = LayerShape(B=s.B, H=s.H, P=s.P, N=s.N, G=s.G, L=s.L, T_max=1, in_dtype=s.in_dtype,
                             read_fmt=read_fmt, ckpt=ckpt, seed=s.seed, recurrence=recurrence)
        self.dev = torch.device("cuda", local)
        self.stream = torch.cuda.current_stream()
        gen = torch.Generator(device=self.dev)
        gen.manual_seed(s.seed + 1000 * rank)
        self.ckpt0 = torch.randn((s.B, s.H, s.P, s.N), generator=gen, device=self.dev, dtype=torch.float32) * 0.1
        self.model = ReplaySSM(self.ls, self.ckpt0.to(self.ls.torch_ckpt_dtype))
        self.pool = decode_pool(s, self.ls, self.dev, gen, self.delta)
        self.out = torch.empty((s.B, s.H, s.P), dtype=torch.float32, device=self.dev)
        self.launches = 0
        # kernels per decode step: the warp-per-head non-flush kernel and the head kernel
        # (read copies, by default), or the head kernel alone
        self.decode_kernels = self.model.decode_kernel()
        self.kernels_per_step = 2 if self.decode_kernels == "warp_per_head" else 1

    static_scratch = False  # decode steps through rssm_decode_step_static_scratch

    def step(self, x, o, st=None):
        if self.static_scratch:
            self.model.decode_step_static_scratch(*x, out=o, stream=st)
        elif self.delta:
            self.model.decode_step(*x[:4], out=o, beta=x[4], stream=st)
        else:
            self.model.decode_step(*x, out=o, stream=st)
        self.launches += 1

    def window(self, i0: int, ev: list | None = None):
        for j in range(self.s.L):
            x = self.pool[(i0 + j) % len(self.pool)]
            if ev is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                self.step(x, self.out)
                e1.record(self.stream)
                ev.append((e0, e1))
            else:
                self.step(x, self.out)

    def warm(self, warmup: int) -> float:
        """warmup whole windows (every sequence stays aligned on the window); returns s per window."""
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.window(0)
        w0.record(self.stream)
        for w in range(1, max(2, warmup)):
            self.window(w * self.s.L)
        w1.record(self.stream)
        torch.cuda.synchronize()
        self.model.read_pointers()  # raises on any device error
        return w0.elapsed_time(w1) / 1e3 / max(1, max(2, warmup) - 1)

    def timed(self, n_windows: int, world: int, clock=None):
        """n_windows timed windows with per-launch events; returns (elapsed s, per-launch s)."""
        evs: list = []
        barrier(world)
        torch.cuda.synchronize()
        ctx = clock if clock is not None else _Null()
        with ctx:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(self.stream)
            for i in range(n_windows):
                self.window(i * self.s.L, evs)
            t1.record(self.stream)
            torch.cuda.synchronize()
        barrier(world)
        return t0.elapsed_time(t1) / 1e3, [a.elapsed_time(b) / 1e3 for a, b in evs]

    def roofline(self, launch_s: list, peak: float, peak_kind: str, traffic) -> dict:
        s, L = self.s, self.s.L
        wb = window_bytes(s, self.read_fmt, 4 if self.ckpt_fmt == "f32" else 2, self.delta)
        alg = wb["replay_per_seq_step"] * s.B
        mean = sum(launch_s) / len(launch_s)
        flush_s = [launch_s[i] for i in range(len(launch_s)) if i % L == L - 1]
        nonflush_s = [launch_s[i] for i in range(len(launch_s)) if i % L != L - 1]
        nf = sum(nonflush_s) / max(1, len(nonflush_s))
        fl = sum(flush_s) / max(1, len(flush_s))
        achieved = alg / mean / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": peak_kind, "traffic": traffic, "algorithmic_bytes_per_launch": alg,
                "mean_launch_ms": mean * 1e3, "mean_nonflush_launch_ms": nf * 1e3, "mean_flush_launch_ms": fl * 1e3,
                "nonflush_frac": wb["nonflush_per_seq_launch"] * s.B / nf / 1e9 / peak if nf > 0 else None,
                "flush_frac": wb["flush_per_seq_launch"] * s.B / fl / 1e9 / peak if fl > 0 else None,
                "frac_of_nominal_8tbs": achieved / 8000.0}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False

    def summary(self):
        return None


def windows_for(args_steps: int, per_window_s: float, min_seconds: float) -> int:
    """Timed windows: at least --steps, and enough to fill min_seconds."""
    return max(args_steps, int(math.ceil(min_seconds / max(per_window_s, 1e-6))))


def run_ours(args, world, rank, local):
    from hybrid_model_ssm_gb300 import conventional_step

    torch.cuda.set_device(local)
    s = WORKLOAD if args.batch is None else WORKLOAD.with_(B=args.batch)
    delta = args.recurrence == "delta"
    arm = DecodeArm(s, local, rank, args.read_fmt, args.ckpt, args.recurrence)
    L = s.L
    per_window = arm.warm(args.warmup)
    n_windows = windows_for(args.steps, per_window, args.min_seconds)
    with ClockSampler(local) as clk:
        elapsed, launch_s = arm.timed(n_windows, world, clk)
    timed_launches = len(launch_s) * arm.kernels_per_step
    decode_kernels = arm.decode_kernels
    start, count, err = arm.model.read_pointers()
    elapsed_max = max_over_ranks(elapsed, world)
    seq_steps = world * s.B * L * n_windows
    value = seq_steps / elapsed_max
    peak, peak_kind = measured_peak_gbs()
    default_case = not (args.read_fmt or args.ckpt != "f32" or args.batch is not None)
    traffic = (profiled_traffic("delta_decode_b256_l16" if delta else "decode_b256_l16") if default_case else None)
    roof = arm.roofline(launch_s, peak, peak_kind, traffic)
    ckpt_es = 4 if args.ckpt == "f32" else 2
    wb = window_bytes(s, args.read_fmt, ckpt_es, delta)
    model, pool, out, stream = arm.model, arm.pool, arm.out, arm.stream

    # in-run comparison: the conventional kernel on the same workload
    comp = None
    if not args.no_conventional:
        state = arm.ckpt0.clone()
        n_conv = max(1, min(n_windows, 50))

        def conv(x):
            conventional_step(arm.ls, state, *x[:4], out=out, beta=x[4] if delta else None)

        for i in range(L):
            conv(pool[i % len(pool)])
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(n_conv * L):
            conv(pool[i % len(pool)])
        c1.record(stream)
        torch.cuda.synchronize()
        conv_t = c0.elapsed_time(c1) / 1e3
        conv_value = s.B * L * n_conv / conv_t
        conv_bytes = wb["conventional_per_seq_step"] * s.B * L * n_conv
        comp = {"conventional_seq_steps_per_s": conv_value,
                "conventional_hbm_gbs": conv_bytes / conv_t / 1e9,
                "replay_speedup": value / world / conv_value,
                "replay_state_bytes_per_window_over_conventional": (L + 1) / (2 * L) * ckpt_es / 4,
                "windows_timed": n_conv}
        del state

    # End to end through the public API with host buffers: every decode step's
    # inputs come from pinned host memory and its output goes back to it. The
    # copies run on two copy streams (in, out) and the decode steps on the
    # compute stream, with double-buffered device inputs and outputs, so step
    # t's kernel overlaps step t+1's input copy and step t-1's output copy.
    e2e = None
    if not args.no_e2e:
        host_pool = [tuple(x.cpu().pin_memory() for x in step) for step in pool]
        dpool = [tuple(torch.empty_like(x) for x in pool[0]) for _ in range(2)]
        dout = [torch.empty_like(out) for _ in range(2)]
        host_out = [torch.empty((s.B, s.H, s.P), dtype=torch.float32).pin_memory() for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in host_pool[0])
        d2h = host_out[0].numel() * host_out[0].element_size()
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer j landed
        ev_done = [torch.cuda.Event() for _ in range(2)]  # the step on buffer j finished
        ev_out = [torch.cuda.Event() for _ in range(2)]   # output j copied out
        n_e2e = max(1, min(n_windows, 120))
        torch.cuda.synchronize()
        barrier(world)
        tw0 = time.perf_counter()
        for i in range(n_e2e * L):
            j = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(ev_done[j])  # step i-2 has read buffer j
                for d, h in zip(dpool[j], host_pool[i % len(host_pool)]):
                    d.copy_(h, non_blocking=True)
                ev_in[j].record(h2d_s)
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_out[j])  # step i-2's output has been copied out
            arm.step(dpool[j], dout[j], stream)
            ev_done[j].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[j])
                host_out[j].copy_(dout[j], non_blocking=True)
                ev_out[j].record(d2h_s)
        torch.cuda.synchronize()
        tw = max_over_ranks(time.perf_counter() - tw0, world)
        e2e = {"value": world * s.B * L * n_e2e / tw, "unit": UNIT, "h2d_bytes_per_step": h2d * L,
               "d2h_bytes_per_step": d2h * L, "windows_timed": n_e2e,
               "note": "pinned host inputs copied in and outputs copied out every decode step; the copies run "
                       "on an input and an output copy stream, overlapping the neighbouring steps' kernels "
                       "(double-buffered device inputs and outputs)"}
    del arm, model, pool, out
    torch.cuda.empty_cache()

    # the path's other arms, each with its own roofline block (default case only)
    extras = {}
    if default_case and not delta and not args.no_extras:
        extras = secondary_arms(args, world, rank, local)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_line(s, delta=delta)

    if rank != 0:
        return None
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / n_windows * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if args.ckpt == "f32" else "f32 (fp16 checkpoint)",
        "data": "synthetic",
        "config": {"workload": f"ReplaySSM decode, one {'gated delta-rule' if delta else 'Mamba-2-shaped'} layer: "
                               f"B={s.B} H={s.H} P={s.P} N={s.N} "
                               f"G={s.G} L={L}, bf16 v/k/q, fp32 checkpoint and outputs; one step = one window "
                               f"of {L} decode launches ({L - 1} non-flush + 1 flush)",
                   "global_batch": s.B * world, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush needed: the 1 GiB checkpoint per replica is 8x the 129 MB L2",
                   "inputs": "16 resident steps of seeded inputs, cycled",
                   "windows_timed": n_windows,
                   "timed_region": f"max(--steps, enough windows for {args.min_seconds:g} s) = {n_windows} windows"},
        "hbm_gbs_achieved": roof["achieved"],
        "roofline": roof,
        "comparison": comp,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": timed_launches,
        "decode_kernels": decode_kernels,
        "device_error_word": err,
    }
    line.update(extras)
    return line


def secondary_arms(args, world, rank, local) -> dict:
    """The verify rounds, the read-copy, delta-rule and FP16-checkpoint decodes and the
    static-scratch step, each timed for at least --extra-seconds, with the roofline of
    its dominant launch."""
    out = {}
    peak, peak_kind = measured_peak_gbs()
    vargs = argparse.Namespace(**vars(args))
    vargs.batch, vargs.drafts = None, None
    vargs.min_seconds = args.extra_seconds
    for key, rec in (("verify_b512_t4", "outer"), ("delta_verify_b512_t4", "delta")):
        vargs.recurrence = rec
        v = run_verify(vargs, world, rank, local, print_line=False)
        torch.cuda.empty_cache()
        if v is not None:
            out[key] = {k: v[k] for k in ("metric", "value", "unit", "ms_per_step", "verify_kernel", "roofline",
                                          "breakdown_ms_per_round", "comparison", "clocks", "gpu_launches",
                                          "device_error_word") if k in v}
            out[key]["rounds_timed"] = v["config"]["rounds_timed"]
    for key, kw in (("read_copy_e4m3", {"read_fmt": "e4m3"}), ("read_copy_e2m1", {"read_fmt": "e2m1"}),
                    ("delta_rule", {"recurrence": "delta"}), ("ckpt_f16_sr", {"ckpt": "f16_sr"}),
                    ("ckpt_f16_rn", {"ckpt": "f16_rn"})):
        arm = DecodeArm(WORKLOAD, local, rank, **kw)
        per_window = arm.warm(args.warmup)
        n = windows_for(args.steps, per_window, args.extra_seconds)
        with ClockSampler(local) as clk:
            elapsed, launch_s = arm.timed(n, world, clk)
        err = arm.model.read_pointers()[2]
        traffic = profiled_traffic("delta_decode_b256_l16" if key == "delta_rule" else key + "_b256_l16")
        elapsed = max_over_ranks(elapsed, world)
        out[key] = {"value": world * WORKLOAD.B * WORKLOAD.L * n / elapsed, "unit": UNIT,
                    "ms_per_window": elapsed / n * 1e3, "windows_timed": n,
                    "roofline": arm.roofline(launch_s, peak, peak_kind, traffic),
                    "clocks": clk.summary(), "decode_kernels": arm.decode_kernels,
                    "gpu_launches": len(launch_s) * arm.kernels_per_step, "device_error_word": err}
        del arm
        torch.cuda.empty_cache()
    out["static_scratch"] = static_scratch_arm(args, world, rank, local)
    torch.cuda.empty_cache()
    return out


def static_scratch_arm(args, world, rank, local, blocks: int = 4) -> dict:
    """The headline workload stepped through rssm_decode_step_static_scratch (tickets in the
    library's static array, cleared by a memset before every launch) and through
    rssm_decode_step, in alternating blocks of windows on one layer."""
    arm = DecodeArm(WORKLOAD, local, rank)
    per_window = arm.warm(args.warmup)
    n = max(1, windows_for(args.steps, per_window, args.extra_seconds) // blocks)
    t = {False: 0.0, True: 0.0}
    with ClockSampler(local) as clk:
        for b in range(2 * blocks):
            arm.static_scratch = b % 2 == 1
            elapsed, _ = arm.timed(n, world)
            t[arm.static_scratch] += max_over_ranks(elapsed, world)
    err = arm.model.read_pointers()[2]
    units = world * WORKLOAD.B * WORKLOAD.L * n * blocks
    res = {"value": units / t[True], "unit": UNIT, "windows_timed": n * blocks,
           "ms_per_window": t[True] / (n * blocks) * 1e3,
           "decode_step_ms_per_window": t[False] / (n * blocks) * 1e3,
           "decode_step_value": units / t[False], "clocks": clk.summary(),
           "gpu_launches": 2 * n * blocks * WORKLOAD.L * arm.kernels_per_step, "device_error_word": err}
    del arm
    return res


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step is one window of L decode
    steps on a sample of the batch (rank 0 only)."""
    if rank != 0:
        return None
    s = WORKLOAD
    n_seq, threads = 1, host_cores()
    oracle_sample = OracleSample(s, n_seq, threads, seed=s.seed)
    if args.warmup:
        oracle_sample.run(args.warmup * s.L)
    t = oracle_sample.run(args.steps * s.L)
    value = oracle_sample.units(args.steps * s.L) / t
    sample = (f"float64 oracle (conventional recurrence), {threads} threads x {n_seq} sequence (of {s.B}) x "
              f"{s.H} heads, one window of {s.L} decode steps per bench step")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"ReplaySSM decode, B={s.B} H={s.H} P={s.P} N={s.N} G={s.G} L={s.L} "
                                   f"(oracle sample of {threads} x {n_seq} sequences)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": usable_cores(), "threads": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


VERIFY_WORKLOAD = synth.PRESETS["mamba2_verify_b512_t4"]
VERIFY_METRIC = "speculative verify draft-tokens/s at B=512, T=4, L=16 (verify + commit + flush per round)"


def verify_round_bytes(s, T: int, counts: np.ndarray, accepted: np.ndarray, delta: bool = False):
    """Algorithmic HBM bytes of one speculative round for the whole batch.

    verify: per sequence |S| + c|r| + T(|in| + |r| + |o|): the checkpoint once, the
    c committed records, the T drafts' records and queries, T outputs and the T
    appended records. commit: 12 B per sequence. flush: every sequence that
    reaches L records reads |S| and its c records and writes |S| once. A
    delta-rule layer's ring records hold the fp32 pseudo-value w in place of v,
    and its inputs carry beta. Returns (verify_bytes, flush_bytes, counts_after).
    """
    es = 2 if s.in_dtype == "bf16" else 4
    S = 4 * s.H * s.P * s.N
    r = 4 * s.H + (4 if delta else es) * s.H * s.P + es * s.G * s.N  # a ring record
    inp = record_bytes(s, delta) + es * s.G * s.N                    # a draft's inputs
    out = 4 * s.H * s.P
    vb = int(np.sum(S + counts * r + T * (inp + r + out)))
    c2 = counts + accepted
    fl = c2 >= s.L
    fb = int(np.sum(np.where(fl, 2 * S + c2 * r, 0))) + 12 * len(counts)
    return vb, fb, np.where(fl, 0, c2)


def run_verify(args, world, rank, local, print_line: bool = True):
    from hybrid_model_ssm_gb300 import ConventionalVerifier, LayerShape, ReplaySSM

    torch.cuda.set_device(local)
    s = VERIFY_WORKLOAD if args.batch is None else VERIFY_WORKLOAD.with_(B=args.batch)
    if args.drafts is not None:
        s = s.with_(T_max=args.drafts)
    T = s.T_max
    delta = args.recurrence == "delta"
    ls = LayerShape(B=s.B, H=s.H, P=s.P, N=s.N, G=s.G, L=s.L, T_max=T, in_dtype=s.in_dtype,
                    recurrence=args.recurrence)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device=dev)
    gen.manual_seed(s.seed + 1000 * rank)
    model = ReplaySSM(ls, torch.randn((s.B, s.H, s.P, s.N), generator=gen, device=dev) * 0.1)
    model.set_verify_kernel(args.verify_kernel)
    vkernel = model.verify_kernel(T)
    sc = 1.0 / math.sqrt(s.N)
    pool = []
    for _ in range(8):
        u = torch.randn((s.B, T, s.H), generator=gen, device=dev)
        a = torch.exp(-torch.nn.functional.softplus(u)).float()
        v = (torch.randn((s.B, T, s.H, s.P), generator=gen, device=dev) * sc).to(ls.torch_in_dtype)
        k = torch.randn((s.B, T, s.G, s.N), generator=gen, device=dev) * sc
        q = torch.randn((s.B, T, s.G, s.N), generator=gen, device=dev) * sc
        if delta:  # write strengths in (0, 1); unit-norm keys and queries
            beta = torch.sigmoid(torch.randn((s.B, T, s.H), generator=gen, device=dev)).float()
            k, q = k / k.norm(dim=-1, keepdim=True), q / q.norm(dim=-1, keepdim=True)
            pool.append((a, v, k.to(ls.torch_in_dtype), q.to(ls.torch_in_dtype), beta))
        else:
            pool.append((a, v, k.to(ls.torch_in_dtype), q.to(ls.torch_in_dtype)))
    cgen = synth.make_generator(s.seed + 7)
    acc_host: list = []
    acc_dev: list = []

    def draw(n):
        for _ in range(n):
            acc_host.append(synth.accepted_lengths(s.B, T, cgen))
            acc_dev.append(acc_host[-1].to(dev))

    out = torch.empty((s.B, T, s.H, s.P), dtype=torch.float32, device=dev)

    def one_round(i, ev=None):
        x = pool[i % len(pool)]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if ev is not None else None
        if e: e[0].record(stream)
        model.verify(*x[:4], out=out, beta=x[4] if delta else None)
        if e: e[1].record(stream)
        model.commit(acc_dev[i])
        if e: e[2].record(stream)
        model.flush(s.L)
        if e: e[3].record(stream); ev.append(e)

    counts = np.zeros(s.B, np.int64)
    draw(args.warmup)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == 1:
            w0.record(stream)
        one_round(i)
        _, _, counts = verify_round_bytes(s, T, counts, acc_host[i].numpy().astype(np.int64), delta)
    w1.record(stream)
    torch.cuda.synchronize()
    model.read_pointers()
    per_round = w0.elapsed_time(w1) / 1e3 / max(1, args.warmup - 1)
    n_rounds = windows_for(args.steps, per_round, args.min_seconds)
    draw(n_rounds)
    rounds = args.warmup + n_rounds
    ev = []
    vbytes = fbytes = 0
    for i in range(args.warmup, rounds):
        vb, fb, counts = verify_round_bytes(s, T, counts, acc_host[i].numpy().astype(np.int64), delta)
        vbytes += vb
        fbytes += fb
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.warmup, rounds):
            one_round(i, ev)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    _, count_dev, err = model.read_pointers()
    assert np.array_equal(count_dev.numpy(), counts), "host pointer replay diverged from the device"
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, world)
    tv = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    tc = sum(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    tf = sum(e[2].elapsed_time(e[3]) for e in ev) / 1e3
    peak, peak_kind = measured_peak_gbs()
    achieved = vbytes / tv / 1e9

    # in-run comparison: conventional verify with per-draft snapshots (one state
    # read and T writes per round, commit by slot index), same inputs and accepts
    comp = None
    if not args.no_conventional and T <= 8 and not delta:  # the snapshot comparator: outer product, T <= 8
        del model
        torch.cuda.empty_cache()
        conv = ConventionalVerifier(ls, torch.randn((s.B, s.H, s.P, s.N), generator=gen, device=dev) * 0.1)
        for i in range(args.warmup):
            a, v, k, q = pool[i % len(pool)]
            conv.verify(a, v, k, q, out=out)
            conv.commit(acc_dev[i])
        torch.cuda.synchronize()
        n_conv = min(n_rounds, max(args.steps, 20))
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(args.warmup, args.warmup + n_conv):
            a, v, k, q = pool[i % len(pool)]
            conv.verify(a, v, k, q, out=out)
            conv.commit(acc_dev[i])
        c1.record(stream)
        torch.cuda.synchronize()
        assert int(conv.err.item()) == 0
        ct = c0.elapsed_time(c1) / 1e3
        es = 2 if s.in_dtype == "bf16" else 4
        Sb = 4 * s.H * s.P * s.N
        inp = record_bytes(s) + es * s.G * s.N
        conv_round = s.B * ((1 + T) * Sb + T * (inp + 4 * s.H * s.P)) + 8 * s.B
        replay_per_round = elapsed / n_rounds
        comp = {"conventional_draft_tokens_per_s": s.B * T * n_conv / ct,
                "conventional_ms_per_round": ct / n_conv * 1e3,
                "conventional_hbm_gbs": conv_round * n_conv / ct / 1e9,
                "replay_speedup": (ct / n_conv) / replay_per_round,
                "algorithmic_bytes_replay_over_conventional": (vbytes + fbytes) / n_rounds / conv_round,
                "rounds_timed": n_conv,
                "method": "every draft advances the full fp32 state and writes a snapshot; commit selects the "
                          "accepted snapshot by a per-sequence slot index"}
        del conv
    if rank != 0:
        return None
    return {
        "metric": VERIFY_METRIC, "value": world * s.B * T * n_rounds / elapsed, "unit": "draft-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / n_rounds * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"ReplaySSM speculative round{' (gated delta-rule layer)' if delta else ''}: "
                               f"B={s.B} H={s.H} P={s.P} N={s.N} G={s.G} L={s.L} "
                               f"T={T}, bf16 inputs; one step = verify + commit (seeded accepted lengths "
                               f"0..{T}) + flush of sequences at {s.L} records",
                   "global_batch": s.B * world, "l2": "no flush needed: 2 GiB checkpoint per replica",
                   "rounds_timed": n_rounds},
        "seq_rounds_per_s": world * s.B * n_rounds / elapsed,
        "verify_kernel": vkernel,
        "roofline": {"bound": "hbm", "kernel": f"verify ({vkernel.replace('_', ' ')})", "achieved": achieved,
                     "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": (profiled_traffic(f"{'delta_' if delta else ''}verify_b512_t{T}")
                                 if args.batch is None else None),
                     "algorithmic_bytes_per_launch": vbytes / n_rounds,
                     "mean_launch_ms": tv / n_rounds * 1e3},
        "breakdown_ms_per_round": {"verify": tv / n_rounds * 1e3, "commit": tc / n_rounds * 1e3,
                                   "flush": tf / n_rounds * 1e3,
                                   "flush_hbm_gbs": fbytes / tf / 1e9 if tf > 0 else None},
        "comparison": comp,
        "clocks": clk.summary(), "gpu_launches": 4 * n_rounds,  # verify, commit, flush list, flush
        "device_error_word": err,
    }


MULTI_SHAPES = {"mamba2": synth.PRESETS["mamba2_layer_b256_l16"], "alt": synth.PRESETS["alt_h32_p128_n128_g16"]}


def run_multilayer(args, world, rank, local):
    """A stack of SSM layers: every decode step runs all layers in turn.

    Sweeps batch and window. Per point: the time of one decode step over all
    layers (CUDA events; launched one by one, and replayed from a CUDA graph
    captured over one step of all layers), the algorithmic HBM bytes of that
    step (window average) and the bandwidth they imply. The per-CTA layout
    choice is made on the device, so a captured step stays valid at every
    window position and the graph is captured once.
    """
    from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM, workspace_size

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    base = MULTI_SHAPES[args.shape]
    batches = [int(x) for x in args.batches.split(",")]
    windows = [int(x) for x in args.windows.split(",")]
    n_layers = args.layers
    peak, peak_kind = measured_peak_gbs()
    points = []
    total_launches = 0
    with ClockSampler(local) as clk:
        for L in windows:
            for B in batches:
                s = base.with_(B=B, L=L)
                ls = LayerShape(B=B, H=s.H, P=s.P, N=s.N, G=s.G, L=L, T_max=1, in_dtype=s.in_dtype)
                ring_b, ptr_b, _ = workspace_size(ls)
                state_b = B * s.H * s.P * s.N * 4
                need = n_layers * (state_b + ring_b + ptr_b + 4 * B * s.H * s.P)
                free, _ = torch.cuda.mem_get_info()
                if need > 0.85 * free:
                    points.append({"B": B, "L": L, "skipped": f"needs {need / 2**30:.1f} GiB, {free / 2**30:.1f} free"})
                    continue
                gen = torch.Generator(device=dev)
                gen.manual_seed(s.seed + 1000 * rank + 17 * L + B)
                models = [ReplaySSM(ls, torch.randn((B, s.H, s.P, s.N), generator=gen, device=dev) * 0.1)
                          for _ in range(n_layers)]
                sc = 1.0 / math.sqrt(s.N)
                pool = []
                for _ in range(4):
                    u = torch.randn((B, s.H), generator=gen, device=dev)
                    pool.append((torch.exp(-torch.nn.functional.softplus(u)).float(),
                                 (torch.randn((B, s.H, s.P), generator=gen, device=dev) * sc).to(ls.torch_in_dtype),
                                 (torch.randn((B, s.G, s.N), generator=gen, device=dev) * sc).to(ls.torch_in_dtype),
                                 (torch.randn((B, s.G, s.N), generator=gen, device=dev) * sc).to(ls.torch_in_dtype)))
                outs = [torch.empty((B, s.H, s.P), dtype=torch.float32, device=dev) for _ in range(n_layers)]

                def step(i):
                    a, v, k, q = pool[i % len(pool)]
                    for m, o in zip(models, outs):
                        m.decode_step(a, v, k, q, out=o)

                for i in range(max(L, args.warmup)):  # every layer has flushed once
                    step(i)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for i in range(args.steps):
                    step(i)
                e1.record(stream)
                torch.cuda.synchronize()
                t_eager = e0.elapsed_time(e1) / 1e3 / args.steps
                # one step of all layers as a CUDA graph, replayed
                graph = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    with torch.cuda.graph(graph, stream=side):
                        step(0)
                stream.wait_stream(side)
                for _ in range(L):
                    graph.replay()
                torch.cuda.synchronize()
                g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                g0.record(stream)
                for _ in range(args.steps):
                    graph.replay()
                g1.record(stream)
                torch.cuda.synchronize()
                t_graph = g0.elapsed_time(g1) / 1e3 / args.steps
                errs = [m.read_pointers()[2] for m in models]
                total_launches += n_layers * (2 * args.steps + max(L, args.warmup) + 1 + L)
                step_bytes = n_layers * B * window_bytes(s)["replay_per_seq_step"]
                points.append({
                    "B": B, "L": L, "ms_per_step": t_eager * 1e3, "ms_per_step_graph": t_graph * 1e3,
                    "seq_steps_per_s_graph": B / t_graph, "algorithmic_bytes_per_step": step_bytes,
                    "hbm_gbs": step_bytes / t_eager / 1e9, "hbm_gbs_graph": step_bytes / t_graph / 1e9,
                    "frac_graph": step_bytes / t_graph / 1e9 / peak,
                    "state_bytes_all_layers": n_layers * state_b,
                    "l2_may_hold_state": n_layers * state_b < 129e6,
                    "device_error_words": sorted(set(errs))})
                del graph, models, pool, outs
                torch.cuda.empty_cache()
    if rank != 0:
        return None
    return {
        "metric": f"multi-layer decode step time ({n_layers} layers), batch x window sweep", "unit": "ms/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{n_layers} SSM layers of H={base.H} P={base.P} N={base.N} G={base.G}, bf16 v/k/q, "
                               f"fp32 checkpoints; one step = one decode step through every layer; inputs: 4 "
                               f"resident steps shared by the layers",
                   "batches": batches, "windows": windows,
                   "l2": "state of all layers vs the 129 MB L2 is given per point (l2_may_hold_state)"},
        "peak_gbs": peak, "peak_kind": peak_kind, "points": points, "clocks": clk.summary(),
        "gpu_launches": total_launches,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300, help="timed windows of L decode steps")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-conventional", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (smaller cases for ncu captures; not a bench line)")
    ap.add_argument("--workload", choices=["decode", "verify", "multilayer"], default="decode",
                    help="decode: the headline metric; verify: speculative rounds (B=512, T=4); "
                         "multilayer: a stack of layers, batch x window sweep (--steps = decode steps per point)")
    ap.add_argument("--layers", type=int, default=40, help="multilayer: layers in the stack")
    ap.add_argument("--shape", choices=sorted(MULTI_SHAPES), default="mamba2",
                    help="multilayer: mamba2 (H=128 P=64 N=128 G=8) or alt (H=32 P=128 N=128 G=16)")
    ap.add_argument("--batches", default="1,32,128,256,512", help="multilayer: batch sizes")
    ap.add_argument("--windows", default="4,8,16,32", help="multilayer: windows L")
    ap.add_argument("--read-fmt", choices=["e4m3", "e2m1"], default=None,
                    help="non-flush steps read a low-precision copy of the checkpoint")
    ap.add_argument("--ckpt", choices=["f32", "f16_sr", "f16_rn"], default="f32",
                    help="checkpoint storage: FP32, or FP16 stored with stochastic / nearest rounding")
    ap.add_argument("--drafts", type=int, default=None,
                    help="verify: drafts per round T (1..16; default 4); other values are not the headline config")
    ap.add_argument("--recurrence", choices=["outer", "delta"], default="outer",
                    help="decode: the gated outer-product recurrence or the gated delta rule (beta inputs)")
    ap.add_argument("--verify-kernel", choices=["auto", "cuda_cores", "tensor_cores"], default="auto",
                    help="verify: the kernel of the verify launches (auto: CUDA cores up to 8 drafts, tensor "
                         "cores above)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="the timed region covers at least this long (and at least --steps steps)")
    ap.add_argument("--extra-seconds", type=float, default=0.3,
                    help="timed length of each secondary arm of the default line")
    ap.add_argument("--no-clocks", action="store_true",
                    help="do not sample clocks with nvidia-smi (profiler runs)")
    ap.add_argument("--no-extras", action="store_true",
                    help="leave out the secondary arms (verify, read copies, delta rule, FP16 checkpoints, static scratch) of the default line")
    args = ap.parse_args(argv)
    if args.recurrence == "delta" and (args.workload == "multilayer" or args.read_fmt or args.ckpt != "f32"):
        ap.error("--recurrence delta: decode or verify workload, FP32 checkpoint, no read copy")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ClockSampler.enabled = not args.no_clocks
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU (there is no CPU fallback)")
        run = {"decode": run_ours, "verify": run_verify, "multilayer": run_multilayer}[args.workload]
        line = run(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
