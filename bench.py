#!/usr/bin/env python
"""Throughput of the causal kernelised linear-attention forward on GB300.

Default workload: B=2, H=16, N=32768, d=dv=64, bf16 q/k/v ~ N(0,1), elu+1
feature map, normalised, causal -- one "step" is one la_forward over the
whole batch (every step of the hot path: feature map, chunk states, chunk
scan, intra- and inter-chunk products, normalisation).  Prints ONE JSON line
on rank 0 with token*heads/s, the roofline fraction of the dominant kernel,
an end-to-end figure through the C ABI with host buffers, and the fp64
oracle timed on the host cores as a CPU baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent sequences: weak scaling, no data-path collective); the timed
region is bracketed by barriers and the max over ranks is reported.
`--impl reference` times the fp64 CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
METRIC = "causal linear-attn fwd token·heads/s at N=32768,d=64; % of HBM/TC roofline"
UNIT = "token*heads/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 10**6

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="causal_n32768_d64_bf16")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def load_peaks():
    path = ROOT / "MEASURED_PEAKS.json"
    if path.exists():
        d = json.loads(path.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (every rank gets it); x itself on one rank."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: int, world: int, steps: int, ms_total: float) -> float:
    """Whole-job units per second: every rank processes units_per_step per
    step (weak scaling), the job takes the slowest rank's time."""
    return units_per_step * world * steps / (ms_total / 1e3)


# summary file name under profiles/ for the kernels of a path
PROFILE_NAME = {"k_tg_state+k_tg_scan+k_tg_out": "k_tg",
                "k_favor+k_tg_state+k_tg_scan+k_tg_out": "k_favor_tg",
                "k_gla_state+k_gla_scan+k_gla_out": "k_gla"}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of `kernel` on `workload`, from the
    ncu summary under profiles/, or None when there is none or a kernel
    source has changed since it was taken (the summary records the SHA-256 of
    every source file it measured)."""
    import hashlib
    import re

    path = ROOT / "profiles" / f"{kernel}_{workload}_counters.md"
    if not path.exists():
        return None
    text = path.read_text()
    srcs = re.findall(r"^source: (\S+) sha256 ([0-9a-f]{64})$", text, re.M)
    m_tr = re.search(r"^traffic_bytes_per_launch: (\d+)$", text, re.M)
    if not srcs or not m_tr:
        return None
    for name, digest in srcs:  # every source the summary measured is unchanged
        src = ROOT / name
        if not src.exists() or hashlib.sha256(src.read_bytes()).hexdigest() != digest:
            return None
    return int(m_tr.group(1))


# ------------------------------------------------------------ clocks -----
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)], stdout=self.file,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in Path(self.file.name).read_text().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------- workload glue ---
def algorithmic_bytes(w) -> int:
    """Bytes the method must move per forward launch: q, k, v in, fp32 o out
    (the state never needs to leave the chip)."""
    eb = torch.tensor([], dtype=w.dtype).element_size()
    return w.BH * w.N * (2 * w.d * eb + w.dv * eb + w.dv * 4)


def algorithmic_flops(w) -> int:
    """4 r dv + 4 r FLOPs per token and head: rank-1 state update, read, and
    the normaliser update and dot (r = d)."""
    return w.BH * w.N * (4 * w.d * w.dv + 4 * w.d)


def decode_bytes(w) -> int:
    eb = torch.tensor([], dtype=w.dtype).element_size()
    per = 2 * 4 * (w.d * w.dv + w.d) + (2 * w.d + w.dv) * eb + w.dv * 4
    return w.BH * per


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_forward_sample(w, q, k, v, cores):
    """Time the fp64 oracle on whole sequences of the workload (a bounded
    sample); returns (token*heads/s, description, threads)."""
    import numpy as np

    import oracle

    orc = oracle.load()
    ns = min(w.BH, 2 * cores)
    qf, kf, vf = (t.reshape(w.BH, 1, w.N, -1)[:ns].float().cpu().numpy().astype(np.float64)
                  for t in (q, k, v))
    gamma = w.gamma()
    t0 = time.perf_counter()
    alpha = None
    if w.extra.get("gla_gates"):
        from kernelised_causal_linear_gb300 import synth

        lo, hi = w.extra["gla_gates"]
        alpha = synth.gates((w.B, w.H, w.N, w.d), seed=w.seed(31), lo=lo, hi=hi)
        alpha = alpha.reshape(w.BH, 1, w.N, w.d)[:ns].double().numpy()
    if w.extra.get("favor_r"):  # the features are part of the method here
        from kernelised_causal_linear_gb300 import synth

        W = synth.gaussian_rows(w.extra["favor_r"], w.d, seed=w.seed(30)).double().numpy()
        qf, kf = orc.favor(qf, W), orc.favor(kf, W)
    orc.forward(qf.reshape(ns, 1, w.N, -1), kf.reshape(ns, 1, w.N, -1),
                vf.reshape(ns, 1, w.N, -1), causal=w.causal, fm=w.feature_map,
                gamma=None if gamma is None else gamma[:1].double().numpy(), alpha=alpha,
                nthreads=cores)
    dt = time.perf_counter() - t0
    return ns * w.N / dt, f"{ns} of {w.BH} sequences x {w.N} tokens (fp64 oracle)", min(ns, cores), dt


# --------------------------------------------------------------- main ----
def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from kernelised_causal_linear_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    decode = w.steps > 0
    steps = args.steps if args.steps is not None else (200 if decode else 400)
    warmup = args.warmup if args.warmup is not None else 10
    if warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, w, steps, warmup, world)

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    import kernelised_causal_linear_gb300 as la

    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()

    if decode:
        from kernelised_causal_linear_gb300 import prefill

        S, z = prefill.prefill_decode_state(w)
        # a fresh token for every step (cycled after n_tok distinct ones)
        n_tok = min(256, steps + warmup)
        tq, tk, tv = synth.decode_tokens(w, n_tok, device="cuda")
        q, k, v = tq[0], tk[0], tv[0]
        out = torch.empty((w.B, w.H, w.dv), dtype=torch.float32, device="cuda")
        tok_i = [0]

        def step():
            i = tok_i[0] % n_tok
            tok_i[0] += 1
            la.la_decode_step(S, z, tq[i], tk[i], tv[i], out, feature_map=w.feature_map)

        units_per_step = w.BH
        bytes_per_launch = decode_bytes(w)
    elif w.extra.get("gla_gates"):
        # per-key-channel decay: the gates are an input of the method
        q, k, v = synth.qkv(w, device="cuda")
        lo, hi = w.extra["gla_gates"]
        alpha = synth.gates((w.B, w.H, w.N, w.d), seed=w.seed(31), lo=lo, hi=hi, device="cuda")
        out = torch.empty((w.B, w.H, w.N, w.dv), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(16, la.la_gla_workspace_size(w.B, w.H, w.N, w.d, w.dv)),
                         dtype=torch.uint8, device="cuda")

        def call(q_, k_, v_, o_):
            la.la_forward_gla(q_, k_, v_, alpha, o_, feature_map=w.feature_map, workspace=ws)

        def step():
            call(q, k, v, out)

        units_per_step = w.BH * w.N
        bytes_per_launch = algorithmic_bytes(w) + w.BH * w.N * w.d * 4  # + the fp32 gates
    elif w.extra.get("favor_r"):
        # Performer: positive random features of q and k, then the
        # identity-normalised forward over them (feature dimension r)
        r = w.extra["favor_r"]
        q, k, v = synth.qkv(w, device="cuda")
        W = synth.gaussian_rows(r, w.d, seed=w.seed(30), device="cuda")
        fq = torch.empty((w.B, w.H, w.N, r), dtype=w.dtype, device="cuda")
        fk = torch.empty_like(fq)
        out = torch.empty((w.B, w.H, w.N, w.dv), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(16, la.la_forward_workspace_size(w.B, w.H, w.N, r, w.dv, w.causal,
                                                               w.dtype)),
                         dtype=torch.uint8, device="cuda")

        def call(q_, k_, v_, o_):
            la.la_favor_features(q_, W, fq)
            la.la_favor_features(k_, W, fk)
            la.la_forward(fq, fk, v_, o_, causal=w.causal, feature_map="identity_norm",
                          workspace=ws)

        def step():
            call(q, k, v, out)

        units_per_step = w.BH * w.N
        bytes_per_launch = algorithmic_bytes(w)
    else:
        q, k, v = synth.qkv(w, device="cuda")
        out = torch.empty((w.B, w.H, w.N, w.dv), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(16, la.la_forward_workspace_size(w.B, w.H, w.N, w.d, w.dv, w.causal,
                                                               w.dtype)),
                         dtype=torch.uint8, device="cuda")
        gamma = w.gamma()

        def call(q_, k_, v_, o_):
            la.la_forward(q_, k_, v_, o_, causal=w.causal, feature_map=w.feature_map,
                          gamma=gamma, workspace=ws)

        def step():
            call(q, k, v, out)

        units_per_step = w.BH * w.N
        bytes_per_launch = algorithmic_bytes(w)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        barrier()
        torch.cuda.synchronize()
        n0 = la.la_launch_count()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        n1 = la.la_launch_count()
        barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, "cuda")
    ms_step = ms_total / steps
    value = job_throughput(units_per_step, world, steps, ms_total)
    assert la.la_get_device_status() == 0

    # --- end to end through the C ABI with pinned host buffers ------------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(la, w, decode, steps, stream, world, out, locals())

    # --- CPU baseline: the fp64 oracle on a bounded sample -----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        if decode:
            cpu = cpu_decode_baseline(w, S, z, cores)
        else:
            val, desc, used, dt = oracle_forward_sample(w, q, k, v, cores)
            cpu = {"value": val, "unit": UNIT, "cores": used, "kind": "oracle",
                   "sample": f"{desc}; {dt:.1f} s wall"}

    achieved = bytes_per_launch / (ms_step / 1e3) / 1e9
    fdim = w.extra.get("favor_r", w.d)
    path = "decode" if decode else la.la_forward_path(w.B, w.H, w.N, fdim, w.dv, w.causal,
                                                      w.feature_map, w.decay, w.dtype)
    # the kernel(s) one step launches; for the multi-kernel paths the roofline
    # is that of the whole call (every launch of the step inside the time)
    kernel = {"tcgen05": "k_fwd_tc64", "tcgen05_chunked": "k_tg_state+k_tg_scan+k_tg_out",
              "simt": "k_chunk_state+k_block_scan+k_block_out",
              "decode": "k_decode_step"}[path]
    if w.extra.get("favor_r"):
        kernel = "k_favor+" + kernel
    if w.extra.get("gla_gates"):
        # bf16 at d = 128: warp-level tensor-core products; fp32 products otherwise
        path = "gla_mma" if (w.dtype == torch.bfloat16 and w.d == 128) else "gla_fp32"
        kernel = "k_gla_state+k_gla_scan+k_gla_out"
    if decode:
        metric = "batched decode step token*heads/s, d=dv=128"
    elif w.name == "causal_n32768_d64_bf16":
        metric = METRIC
    else:
        metric = f"linear-attn fwd token*heads/s on {w.name}"
    line = {
        "metric": metric,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": la_path_dtype(w),
        "data": "synthetic: seeded i.i.d. normal inputs rounded once to the input dtype",
        "config": {
            "workload": w.name, "B": w.B, "H": w.H, "N": w.N if not decode else 1,
            "d": w.d, "dv": w.dv, "input_dtype": str(w.dtype).replace("torch.", ""),
            "causal": w.causal, "feature_map": w.feature_map, "decay": w.decay,
            "l2": f"no flush: every step moves {bytes_per_launch / 1e6:.0f} MB, more than the "
                  f"{L2_BYTES / 1e6:.0f} MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"],
            "traffic": profiled_traffic(PROFILE_NAME.get(kernel, kernel), w.name),
            "kernel": kernel,
            "path": path,
            "peak_source": f"{peak_src} HBM copy bandwidth",
            "algorithmic_bytes_per_launch": bytes_per_launch,
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(n1 - n0),
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def la_path_dtype(w) -> str:
    """Arithmetic type of the path that runs: bf16 tensor-core operands with
    fp32 accumulation on the tcgen05 kernels and on the GLA products for bf16
    inputs at d = 128, fp32 on the CUDA-core paths."""
    if w.extra.get("gla_gates"):
        return "bf16" if (w.dtype == torch.bfloat16 and w.d == 128) else "f32"
    if w.steps > 0:
        return "f32"
    import kernelised_causal_linear_gb300 as la

    path = la.la_forward_path(w.B, w.H, w.N, w.extra.get("favor_r", w.d), w.dv, w.causal,
                              w.feature_map, w.decay, w.dtype)
    return "bf16" if path.startswith("tcgen05") else "f32"


def run_e2e(la, w, decode, steps, stream, world, out, env):
    """The same metric with host buffers: every step copies its inputs from
    pinned host memory, runs the C-ABI call and reads the result back.
    Consecutive steps use two device buffer sets so that one step's copies
    overlap another step's computation."""
    if decode:
        q, k, v = env["q"], env["k"], env["v"]
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        S, z = env["S"], env["z"]
        # the state stays on the device; the tokens of one step go up and the
        # outputs of the previous one come down while a step runs
        sets = [(q, k, v, out), tuple(torch.empty_like(t) for t in (q, k, v, out))]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        free = [None, None]

        def step(i):
            b = i & 1
            dq, dk, dv, do = sets[b]
            with torch.cuda.stream(s_in):
                if free[b] is not None:
                    s_in.wait_event(free[b])
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            with torch.cuda.stream(stream):
                la.la_decode_step(S, z, dq, dk, dv, do, feature_map=w.feature_map)
                done = torch.cuda.Event()
                done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                hout.copy_(do, non_blocking=True)
                free[b] = torch.cuda.Event()
                free[b].record(s_out)

        units = w.BH
        n = max(3, min(steps, 50))
        for i in range(3):
            step(i)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(s_in)
        for i in range(n):
            step(i)
        ev1.record(s_out)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        if world > 1:
            t = torch.tensor([ms], device="cuda")
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
    else:
        q, k, v = env["q"], env["k"], env["v"]
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        gamma = w.gamma()
        # Two device buffer sets so that the copies of one step overlap the
        # computation of the next: inputs go up on one stream, results come
        # down on another, the forward runs on the bench stream.
        sets = [(q, k, v, out), tuple(torch.empty_like(t) for t in (q, k, v, out))]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        free = [None, None]
        units = w.BH * w.N

        def step(i):
            b = i & 1
            dq, dk, dv, do = sets[b]
            with torch.cuda.stream(s_in):
                if free[b] is not None:
                    s_in.wait_event(free[b])
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            with torch.cuda.stream(stream):
                env["call"](dq, dk, dv, do)
                done = torch.cuda.Event()
                done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                hout.copy_(do, non_blocking=True)
                free[b] = torch.cuda.Event()
                free[b].record(s_out)

        n = max(3, min(steps, 50))
        for i in range(3):
            step(i)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(s_in)
        for i in range(n):
            step(i)
        ev1.record(s_out)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        if world > 1:
            t = torch.tensor([ms], device="cuda")
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = hout.numel() * hout.element_size()
        return {"value": units * world * n / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n,
                "overlap": "the copies of one step overlap the forward of the next"}
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()
    return {"value": units * world * n / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n,
            "overlap": "the copies of one step overlap the decode step before it"}


def cpu_decode_baseline(w, S, z, cores):
    import numpy as np

    import oracle
    from kernelised_causal_linear_gb300 import synth

    orc = oracle.load()
    ns = min(w.BH, 256)
    steps = 5
    Sh = S.reshape(w.BH, 1, w.d, w.dv)[:ns].double().cpu().numpy()
    zh = z.reshape(w.BH, 1, w.d)[:ns].double().cpu().numpy()
    q, k, v = synth.decode_tokens(w, steps, device="cpu")
    qs = q.reshape(steps, w.BH, 1, w.d)[:, :ns].double().numpy()
    ks = k.reshape(steps, w.BH, 1, w.d)[:, :ns].double().numpy()
    vs = v.reshape(steps, w.BH, 1, w.dv)[:, :ns].double().numpy()
    t0 = time.perf_counter()
    for t in range(steps):
        _, Sh, zh = orc.decode_step(Sh, zh, qs[t], ks[t], vs[t], nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": ns * steps / dt, "unit": UNIT, "cores": min(cores, ns), "kind": "oracle",
            "sample": f"{ns} of {w.BH} sequences x {steps} decode steps (fp64 oracle); "
                      f"{dt:.1f} s wall"}


def run_reference(args, w, steps, warmup, world):
    """--impl reference: the fp64 oracle on the host cores, each step a
    bounded sample of the same workload."""
    import numpy as np

    import oracle
    from kernelised_causal_linear_gb300 import synth

    orc = oracle.load()
    cores = cpu_cores()
    gamma = w.gamma()
    if w.steps > 0:
        ns = min(w.BH, 4 * cores)
        Sh = np.zeros((ns, 1, w.d, w.dv))
        zh = np.zeros((ns, 1, w.d))
        q, k, v = synth.decode_tokens(w, 1, device="cpu")
        qs, ks, vs = (t.reshape(w.BH, 1, -1)[:ns].double().numpy() for t in (q[0], k[0], v[0]))

        def step():
            nonlocal Sh, zh
            _, Sh, zh = orc.decode_step(Sh, zh, qs, ks, vs, nthreads=cores)

        units = ns
        desc = f"{ns} of {w.BH} sequences, one decode step each (fp64 oracle)"
    else:
        ns = min(w.BH, cores)
        n_tok = min(w.N, 4096)
        q, k, v = synth.qkv(w, device="cpu", B=1, H=ns, N=n_tok)
        qf, kf, vf = (t.double().numpy() for t in (q, k, v))

        W = (synth.gaussian_rows(w.extra["favor_r"], w.d, seed=w.seed(30)).double().numpy()
             if w.extra.get("favor_r") else None)
        alpha = None
        if w.extra.get("gla_gates"):
            lo, hi = w.extra["gla_gates"]
            alpha = synth.gates((1, ns, n_tok, w.d), seed=w.seed(31), lo=lo, hi=hi).double().numpy()

        def step():
            a, b = (orc.favor(qf, W), orc.favor(kf, W)) if W is not None else (qf, kf)
            orc.forward(a, b, vf, causal=w.causal, fm=w.feature_map,
                        gamma=None if gamma is None else np.full(ns, float(gamma[0])),
                        alpha=alpha, nthreads=cores)

        units = ns * n_tok
        desc = f"{ns} of {w.BH} sequences x first {n_tok} of {w.N} tokens (fp64 oracle)"
    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    value = units * steps / dt
    line = {
        "impl": "reference",
        "metric": METRIC if w.steps == 0 else "batched decode step token*heads/s, d=dv=128",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dv": w.dv},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, ns), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
