#!/usr/bin/env python3
"""Benchmark of the KDA chunked forward pass on GB300.

One step = one ``kda_fwd`` call over the whole B=8, T=4096, H=16, K=V=128
workload (lower_bound -5, no gate parameters, fp32 final state), inputs
resident in HBM. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step). Under torchrun (N > 1) each
rank runs its own copy of the workload on its GPU (weak scaling, no
collective on the data path); the reference arm runs on rank 0 only.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd tokens/s at B=8,T=4096,H=16; achieved HBM GB/s & % of roofline"
UNIT = "tokens/s"
WORKLOAD = "b8_t4096_h16"
BYTES_PER_TOKEN_HEAD = 4 * 256 + 2 + 256     # q, k, v, g in; beta in; out
FLOPS_PER_CHUNK_HEAD = 3 * 2 * 16 * 128 * 128 + 5 * 2 * 16 * 16 * 128 + 2 * 16 ** 3
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
# the device sources the benchmark's kernel (kda_fwd_tc_kernel) is compiled from: counters taken
# under ncu describe the kernel only while these files are unchanged
KERNEL_SOURCES = ["gated_linear_attention_kda_gb300/csrc/" + f for f in
                  ("kda_fwd_tc.cuh", "kda_common.cuh", "kda_chunk.cuh", "tcgen05.cuh", "ptx.cuh", "kda_debug.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "kda_fwd_tc_kernel.b8_t4096_h16.traffic.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def algorithmic(w, d):
    B, T, H = d["q"].shape[0], d["q"].shape[1], d["q"].shape[2]
    nseq = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    st = nseq * H * 128 * 128
    state_bytes = (st * d["initial_state"].element_size() if d["initial_state"] is not None else 0) + st * 4
    nbytes = BYTES_PER_TOKEN_HEAD * B * T * H + state_bytes
    chunks = B * H * math.ceil(T / 16)
    return nbytes, chunks * FLOPS_PER_CHUNK_HEAD


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self):
        return time.perf_counter()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if t0 - 0.06 <= t <= t1 + 0.06] or [l for (_, l) in self.lines[-3:]]
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus, backend="nccl"):
    """Rank, world size and local rank from the launcher's environment; one GPU per rank
    (``backend="gloo"`` keeps everything on the host, for tests without a GPU)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """The largest ``x`` over all ranks (every rank gets it): a job's time is its slowest rank's."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, steps, seconds):
    """Whole-job tokens/s: every rank runs its own copy of the workload (weak scaling), so the
    job processes ``world * tokens_per_rank`` tokens per step in the slowest rank's time."""
    return world * tokens_per_rank * steps / seconds


def oracle_time(d, nthreads, batch_rows):
    """Time the fp64 oracle on the first ``batch_rows`` rows of the workload."""
    import oracle
    import workloads as W
    sl = lambda x: x[:batch_rows].contiguous()
    bits = {k: W.bf16_bits(sl(d[k])) for k in ("q", "k", "v", "g", "beta")}
    A = None if d["A_log"] is None else d["A_log"].numpy()
    db = None if d["dt_bias"] is None else d["dt_bias"].numpy()
    init = None if d["initial_state"] is None else W.state_f64(sl(d["initial_state"]))
    t0 = time.perf_counter()
    oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bits["beta"], d["scale"], A, db, d["lower_bound"],
               init, None, nthreads=nthreads)
    return time.perf_counter() - t0, batch_rows * d["q"].shape[1]


def cpu_baseline(d):
    import oracle
    oracle.build()
    n = oracle.default_threads()
    B = d["q"].shape[0]
    secs, toks = oracle_time(d, n, 1)
    rows = max(1, min(B, int(10.0 / max(secs, 1e-3))))   # aim at ~10 s of CPU work
    if rows > 1:
        secs, toks = oracle_time(d, n, rows)
    return {"value": toks / secs, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{rows} of {B} batch rows x {d['q'].shape[1]} tokens x {d['q'].shape[2]} heads, "
                      f"fp64 per-token recurrence, {secs:.2f} s"}


def run_reference(args, world, rank):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    import workloads as W
    oracle.build()
    d = W.make(WORKLOAD)
    n = oracle.default_threads()
    for _ in range(args.warmup):
        oracle_time(d, n, 1)
    total_s, total_tok = 0.0, 0
    for _ in range(args.steps):
        s, t = oracle_time(d, n, 1)
        total_s += s
        total_tok += t
    v = total_tok / total_s
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD, "B": 8, "T": 4096, "H": 16, "K": 128, "V": 128,
                       "sample_per_step": "1 of 8 batch rows (4096 tokens x 16 heads)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": n, "kind": "oracle",
                             "sample": "1 of 8 batch rows x 4096 tokens x 16 heads per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    import gated_linear_attention_kda_gb300 as kda
    import workloads as W

    d = W.make(WORKLOAD)
    B, T, H = d["q"].shape[0], d["q"].shape[1], d["q"].shape[2]
    dev = torch.device("cuda", torch.cuda.current_device())
    c = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.empty_like(c["v"])
    fin = torch.empty(B, H, 128, 128, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
                d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"])

    for _ in range(max(3, args.warmup)):
        step()
    kda.check_device_status()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    # per-call CUDA events on the launching stream; ms_per_step is the median call, the mean is kept
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = time.perf_counter()
    e0.record(stream)
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.perf_counter()
    barrier(world)
    per_call = [a.elapsed_time(b) for a, b in ev]
    median_ms = max_over_ranks(statistics.median(per_call), world)
    mean_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    clocks = sampler.stop(t_start, t_end) if rank == 0 else None
    kda.check_device_status()

    # end to end through the host-buffer entry point: H2D inputs, kernel, D2H result, every step
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    hout = torch.empty_like(d["v"]).pin_memory()
    hfin = torch.empty(B, H, 128, 128, dtype=torch.float32).pin_memory()

    def e2e_step():
        kda.fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], d["scale"], hout, pin["A_log"],
                     pin["dt_bias"], d["lower_bound"], pin["initial_state"], hfin, pin["cu_seqlens"], device=dev)

    e2e_steps = max(1, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in ("q", "k", "v", "g", "beta"))
    d2h = hout.numel() * hout.element_size() + hfin.numel() * hfin.element_size()
    ceiling = copy_ceiling(h2d, d2h, dev)

    if rank != 0:
        return
    tokens = B * T
    ms_per_step = median_ms
    value = job_throughput(world, tokens, 1, median_ms / 1e3)
    nbytes, nflops = algorithmic(WORKLOAD, d)
    hbm, tflops, src = peaks()
    achieved = nbytes / (ms_per_step / 1e3) / 1e9
    traffic = None
    try:
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_hash") == kernel_hash():
            traffic = tr["bytes_per_launch"]
    except Exception:
        pass
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "H": H, "K": 128, "V": 128, "lower_bound": -5.0,
                   "gate_params": False, "final_state": "fp32",
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.1f} MB per step, no flush)",
                   "parallelism": f"{world} independent replica(s), one CTA per (sequence, head) state"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "peak_source": src, "algorithmic_bytes_per_launch": nbytes,
                     "tensor_frac": (nflops / (ms_per_step / 1e3) / 1e12) / tflops},
        "cpu_baseline": cpu_baseline(d) if world == 1 or rank == 0 else None,
        "ms_per_step_mean": mean_ms,
        "e2e": {"value": job_throughput(world, tokens, e2e_steps, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copy_ceiling": dict(ceiling, tokens_per_s=tokens / (h2d / (ceiling["h2d_gbs"] * 1e9)
                                                                     + d2h / (ceiling["d2h_gbs"] * 1e9)))},
        "clocks": clocks,
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def copy_ceiling(h2d, d2h, dev):
    """Measured pinned-host <-> device copy rates (one cudaMemcpyAsync each way of the step's own
    byte counts, best of 3): the link's ceiling for the end-to-end number."""
    import torch
    res = {}
    for name, nbytes, to_dev in (("h2d_gbs", h2d, True), ("d2h_gbs", d2h, False)):
        host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        devb = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        best = float("inf")
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            (devb.copy_(host, non_blocking=True) if to_dev else host.copy_(devb, non_blocking=True))
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) / 1e3)
        res[name] = nbytes / best / 1e9
        del host, devb
    return res


def run_launches(n, workload=None, T=None, chunk=16, workspace=False):
    """Run ``n`` forward passes of a workload (default: the benchmark's; ``T`` shortens it;
    ``chunk`` 32 runs the 32-token-chunk kernel; ``workspace`` calls kda_fwd_ws) for profilers."""
    import torch

    import gated_linear_attention_kda_gb300 as kda
    import workloads as W
    name = workload or WORKLOAD
    d = W.make(name, T=T)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    nseq = d["q"].shape[0] if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    sdt = torch.float32 if d["initial_state"] is None else d["initial_state"].dtype
    out = torch.empty_like(c["v"])
    fin = torch.empty(nseq, d["q"].shape[2], 128, 128, dtype=sdt, device="cuda")
    ws = torch.empty(kda.workspace_bytes(nseq, d["q"].shape[2], chunk=chunk), dtype=torch.uint8, device="cuda")
    for _ in range(n):
        args = (c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
                d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"])
        if workspace:
            kda.fwd_ws(*args, chunk=chunk, workspace=ws)
        else:
            kda.fwd(*args, chunk=chunk)
    kda.check_device_status()
    print(f"ran {n} launches of {name} (T={d['q'].shape[1]}, chunk {chunk}, workspace {workspace})")


DECODE_B, DECODE_H = 128, 16   # 2048 fp32 states of 64 KiB: 134 MB, larger than L2


def run_decode(args):
    """Single-token steps (kda_decode) on DECODE_B sequences x DECODE_H heads with fp32 states
    updated in place: one JSON line with tokens/s and the HBM fraction of the step's bytes."""
    import torch

    import gated_linear_attention_kda_gb300 as kda
    import workloads as W
    torch.cuda.set_device(0)
    d = W.make("b2_t128_h8", B=DECODE_B, T=1, H=DECODE_H)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.empty_like(c["v"])
    state = c["initial_state"].clone()

    def step():
        kda.decode(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, state, c["A_log"], c["dt_bias"],
                   d["lower_bound"])

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    kda.check_device_status()
    ms = e0.elapsed_time(e1) / args.steps
    units = DECODE_B * DECODE_H
    nbytes = units * (2 * 128 * 128 * 4 + 5 * 128 * 2 + 2) + DECODE_H * (4 + 128 * 4)
    hbm, _, src = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "KDA decode tokens/s (one token per state, fp32 state in place)", "value": DECODE_B / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": "fp32", "data": "synthetic",
        "config": {"workload": f"decode_b{DECODE_B}_h{DECODE_H}", "B": DECODE_B, "H": DECODE_H, "K": 128, "V": 128,
                   "l2": "states larger than L2 (134 MB), no flush"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_source": src, "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": args.steps}), flush=True)


def run_variant(args):
    """Kernel-only timing of one workload (``--workload``, reshaped by ``--B/--T/--H``), optionally
    with raw q/k normalised in the kernel (``--qk-norm``), 32-token chunks (``--chunk 32``), a
    forced split of the V rows (``--v-split``) or through kda_fwd_ws with a workspace allocated
    before the timed region (``--workspace``): its own JSON line, tokens/s and the HBM fraction of
    the algorithmic bytes. Not the benchmark line."""
    import torch

    import gated_linear_attention_kda_gb300 as kda
    import workloads as W
    torch.cuda.set_device(0)
    name = args.workload or WORKLOAD
    if args.v_split:
        os.environ["KDA_V_SPLIT"] = str(args.v_split)
    d = W.make(name, raw_qk=args.qk_norm, B=args.B, T=args.T, H=args.H)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    B, T, H = d["q"].shape[0], d["q"].shape[1], d["q"].shape[2]
    nseq = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    sdt = torch.float32 if d["initial_state"] is None else d["initial_state"].dtype
    out = torch.empty_like(c["v"])
    fin = torch.empty(nseq, H, 128, 128, dtype=sdt, device="cuda")
    ws_bytes = kda.workspace_bytes(nseq, H, qk_l2norm=args.qk_norm, chunk=args.chunk) if args.workspace else 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def step():
        a = (c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
             d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"])
        if args.workspace:
            kda.fwd_ws(*a, qk_l2norm=args.qk_norm, chunk=args.chunk, workspace=ws)
        else:
            kda.fwd(*a, qk_l2norm=args.qk_norm, chunk=args.chunk)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    kda.check_device_status()
    ms = e0.elapsed_time(e1) / args.steps
    st = nseq * H * 128 * 128
    nbytes = BYTES_PER_TOKEN_HEAD * B * T * H + st * fin.element_size() + (
        st * d["initial_state"].element_size() if d["initial_state"] is not None else 0)
    hbm, _, src = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "KDA fwd tokens/s" + (" with q/k L2-normalised in the kernel" if args.qk_norm else ""),
        "value": B * T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": name, "B": B, "T": T, "H": H, "sequences": nseq,
                                        "qk_l2norm": bool(args.qk_norm), "chunk": args.chunk,
                                        "entry": "kda_fwd_ws" if args.workspace else "kda_fwd",
                                        "workspace_bytes": ws_bytes,
                                        "v_split": args.v_split or kda.plan(nseq * H, torch.cuda.get_device_properties(0).multi_processor_count)[0]},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_source": src, "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--launches", type=int, default=0,
                    help="profiling mode: run this many forward passes of the workload and exit (no timing)")
    ap.add_argument("--decode", action="store_true",
                    help="time single-token steps (kda_decode) instead and print their own JSON line")
    ap.add_argument("--workload", default=None,
                    help="kernel-only timing of another workload (workloads.ORDER) on its own JSON line")
    ap.add_argument("--T", type=int, default=None,
                    help="tokens per batch row instead of the workload's (with --launches: a shorter case for "
                         "profiling; otherwise kernel-only timing of the reshaped workload)")
    ap.add_argument("--B", type=int, default=None, help="batch rows instead of the workload's (kernel-only timing)")
    ap.add_argument("--H", type=int, default=None, help="heads instead of the workload's (kernel-only timing)")
    ap.add_argument("--chunk", type=int, choices=[16, 32], default=16,
                    help="kernel-only timing with 32-token chunks (KDA_FLAG_CHUNK32, the chunk-size ablation)")
    ap.add_argument("--v-split", type=int, choices=[1, 2, 4, 8], default=None,
                    help="kernel-only timing with the V rows of each state split over this many CTAs (KDA_V_SPLIT)")
    ap.add_argument("--workspace", action="store_true",
                    help="kernel-only timing through kda_fwd_ws: a split state's CTAs share each chunk's preparation")
    ap.add_argument("--qk-norm", action="store_true",
                    help="kernel-only timing with raw q/k normalised in the kernel (KDA_FLAG_QK_L2NORM)")
    args = ap.parse_args()
    if args.launches:
        run_launches(args.launches, args.workload, args.T, args.chunk, args.workspace)
        return
    if args.decode:
        run_decode(args)
        return
    if args.workload or args.qk_norm or args.chunk != 16 or args.v_split or args.B or args.H or args.T or args.workspace:
        run_variant(args)
        return
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local = dist_setup(args.gpus)
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
