#!/usr/bin/env python3
"""Benchmark of the batched variable-length exact top-K (DSA indexer top-K).

Default workload: the DSv3.2-like decode batch - 64 rows x 163840 fp32
logits, seq_lens ~U[2048, 163840], top_k = 2048, previous-step hint given
(seeded synthetic inputs from ``workloads``; the pages' real decode captures
are not available).  One step = one ``gbtopk_varlen`` call over the batch.

Timing: W untimed warm-up steps, then exactly K steps timed with CUDA events
on the launching stream, bracketed by barrier + synchronize; inputs rotate
over enough device copies that the bytes touched between two uses of a copy
exceed the 129 MB L2 (no flush needed).  ``value`` = rows/s over all ranks
(max time over ranks).  ``e2e`` repeats the measurement through the public
Python API with pinned host inputs copied in and indices copied out each
step.  ``--impl reference`` times the CPU oracle (rank 0 only).

Multi-GPU: rows are independent, so each rank runs its own batch (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "top-K rows/s and HBM GB/s (% of GB300 peak), k=2048, N=163840/262144 fp32"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes per call from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum summed over the call's kernels, cold cache), keyed by
# workload and the SHA-256 prefix of the kernel source it was taken on;
# reported as null once the kernel source changes.
NCU_TRAFFIC = {
    ("dsv32_decode", "8c7d0aec4c2a1e77"): 23_812_608,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gbtopk", "reference"], default="gbtopk")
    ap.add_argument("--workload", choices=["dsv32_decode", "long_row_sweep_1024"],
                    default="dsv32_decode")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="short run for profilers: warm-up + K steps, no clock sampling, "
                         "no e2e and no CPU leg")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed

def dist_init(n_gpus: int):
    """Returns (rank, world, local_rank); initialises torch.distributed for N>1."""
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ workload

SEQ_DIST = {"dsv32_decode": lambda W: f"U[2048,{W}]",
            "long_row_sweep_1024": lambda W: f"U[{W // 2},{W}]"}


def make_case(name: str, rank: int):
    import workloads
    if name == "dsv32_decode":
        return workloads.dsv32_decode(seed=2000 + 17 * rank)
    return workloads.long_row_sweep(1024, 2048, True, seed=3999 + 17 * rank)


def valid_columns(case):
    """Valid columns per row from the public contract (next_n = cr = 1 here)."""
    W = case.logits.shape[1]
    assert case.next_n == 1 and case.compress_ratio == 1
    return [min(max(int(s), 0), W) for s in case.seq_lens.tolist()]


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_sha() -> str:
    p = os.path.join(ROOT, "sparse_attention_top_gb300", "csrc", "gbtopk_kernels.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


# ------------------------------------------------------------------ oracle leg

def oracle_rows_per_s(case, seconds: float = 10.0, rows_per_step: int = 8):
    import oracle
    import torch
    R = case.logits.shape[0]
    oracle.build()
    t0 = time.perf_counter()
    done = 0
    r = 0
    while time.perf_counter() - t0 < seconds:
        sl = slice(r, r + rows_per_step)
        oracle.topk_varlen(case.logits[sl], case.seq_lens[sl], case.top_k, return_values=False)
        done += case.logits[sl].shape[0]
        r = (r + rows_per_step) % R
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def workload_config(args, case) -> dict:
    """The workload keys of the JSON line's config, shared by both arms."""
    R, W = case.logits.shape
    hinted = case.pre_idx is not None
    return {"workload": f"{args.workload}: {R} rows x {W} fp32, top_k={case.top_k}, "
                        f"seq_lens {SEQ_DIST[args.workload](W)}, hint={'yes' if hinted else 'no'}",
            "rows": R, "width": W, "top_k": case.top_k, "hinted": hinted}


def run_reference(args, rank, world):
    if rank != 0:
        return
    case = make_case(args.workload, 0)
    import oracle
    import torch
    oracle.build()
    R = case.logits.shape[0]
    rows_per_step = 8
    r = 0

    def step():
        nonlocal r
        sl = slice(r, r + rows_per_step)
        oracle.topk_varlen(case.logits[sl], case.seq_lens[sl], case.top_k, return_values=False)
        r = (r + rows_per_step) % R

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    rows = rows_per_step * args.steps
    v = rows / dt
    sample = (f"{rows_per_step} rows of the {args.workload} batch per step "
              f"({R} rows x {case.logits.shape[1]} fp32, k={case.top_k}), single thread")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(args, case),
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg

def run_gbtopk(args, rank, world, local):
    import torch
    import sparse_attention_top_gb300 as gb

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = make_case(args.workload, rank)
    R, W = case.logits.shape
    k = case.top_k
    n_valid = valid_columns(case)
    valid_bytes = 4 * sum(n_valid)
    algo_bytes = valid_bytes + R * k * 4          # valid columns read + indices written
    copies = max(2, -(-3 * L2_BYTES // max(valid_bytes, 1)) + 1)
    logits_d = [case.logits.to(dev) for _ in range(copies)]
    seq_d = case.seq_lens.to(dev)
    hint_d = [case.pre_idx.to(dev) for _ in range(copies)] if case.pre_idx is not None else None
    out = torch.empty(R, k, dtype=torch.int32, device=dev)
    ws = torch.zeros(gb.gbtopk_workspace_bytes(R, W, k, torch.float32), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        gb.gbtopk_varlen(logits_d[i % copies], seq_d, k, hint_d[i % copies] if hint_d else None,
                         1, 1, out, None, False, ws)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    if args.profile:
        for s in range(args.steps):
            step(s)
        torch.cuda.synchronize(dev)
        if rank == 0:
            print(json.dumps({"profile_run": True, "steps": args.steps, "rows": R, "width": W,
                              "algorithmic_bytes_per_launch": algo_bytes}), flush=True)
        return

    # The K timed steps are captured into one CUDA graph (step s runs on
    # input copy s % copies, so the bytes touched between two uses of a copy
    # exceed the L2): replaying it removes the host launch latency, and
    # consecutive calls overlap their launch with the previous call's tail
    # through programmatic dependent launch, as in a decode loop.
    gstream = torch.cuda.Stream(dev)
    gstream.wait_stream(stream)
    with torch.cuda.stream(gstream):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gstream):
            for s_ in range(args.steps):
                step(s_)
    torch.cuda.synchronize(dev)

    def timed(run, n):
        barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        run(n)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return t0.elapsed_time(t1)

    def eager(n):
        for s_ in range(n):
            step(s_)

    # keep the GPU busy ~1 s around the timed region so the clock samples
    # reflect it (untimed replays also serve as warm-up), then time exactly
    # K steps: one replay of the K-step graph
    with ClockSampler(local) as clk:
        t_end = time.perf_counter() + 0.6
        while time.perf_counter() < t_end:
            graph.replay()
        torch.cuda.synchronize(dev)
        total_ms = timed(lambda n: graph.replay(), args.steps)
        t_end = time.perf_counter() + 0.4
        while time.perf_counter() < t_end:
            graph.replay()
        torch.cuda.synchronize(dev)
    eager_ms = timed(eager, args.steps)
    launch_ms = [total_ms / args.steps]
    total_ms_max = reduce_max(total_ms)
    eager_ms_max = reduce_max(eager_ms)
    rows_all = reduce_sum(R * args.steps)
    value = rows_all / (total_ms_max / 1e3)
    avg_launch_s = statistics.mean(launch_ms) / 1e3
    peak, peak_src = peak_hbm()
    achieved = algo_bytes / avg_launch_s / 1e9
    traffic = NCU_TRAFFIC.get((args.workload, kernel_sha()))
    plan = gb.gbtopk_plan_query(R, W, k, torch.float32)
    kernels_per_call = 3 if plan["split"] else 1

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(case, dev, args, gb)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, rows_done, secs = oracle_rows_per_s(case)
        cpu = {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": f"{rows_done} rows of this batch (8 rows per call, cycling), "
                         f"{secs:.1f} s, single thread"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {**workload_config(args, case),
                       "l2": f"inputs rotate over {copies} device copies "
                             f"({copies * valid_bytes / 2**20:.0f} MB valid > L2)",
                       "parallelism": f"replicas x{world} (rows independent)"},
            "gpu_launches": args.steps * kernels_per_call,
            "timing": {"mode": "one CUDA graph of the K steps, replayed once",
                       "kernels_per_call": kernels_per_call,
                       "eager_ms_per_step": eager_ms_max / args.steps},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": algo_bytes,
                         "avg_launch_us": avg_launch_s * 1e6,
                         "kernel": "the whole call (row + stream + finalize kernels)"},
            "clocks": clk.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_e2e(case, dev, args, gb):
    """Same metric through the public API: pinned host inputs copied in and
    indices copied out inside the timed region, every step."""
    import torch
    R, W = case.logits.shape
    k = case.top_k
    h_logits = case.logits.pin_memory()
    h_seq = case.seq_lens.pin_memory()
    h_hint = case.pre_idx.pin_memory() if case.pre_idx is not None else None
    h_out = torch.empty(R, k, dtype=torch.int32).pin_memory()
    d_logits = torch.empty_like(h_logits, device=dev)
    d_seq = torch.empty_like(h_seq, device=dev)
    d_hint = torch.empty_like(h_hint, device=dev) if h_hint is not None else None
    d_out = torch.empty(R, k, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        d_logits.copy_(h_logits, non_blocking=True)
        d_seq.copy_(h_seq, non_blocking=True)
        if d_hint is not None:
            d_hint.copy_(h_hint, non_blocking=True)
        gb.top_k_varlen(d_logits, d_seq, k, pre_idx=d_hint, out_indices=d_out)
        h_out.copy_(d_out, non_blocking=True)

    steps = max(10, min(args.steps, 50))
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max(a.elapsed_time(b))
    rows = reduce_sum(R * steps)
    h2d = h_logits.numel() * 4 + h_seq.numel() * 4 + (h_hint.numel() * 4 if h_hint is not None else 0)
    return {"value": rows / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": R * k * 4, "steps": steps}


def main():
    args = parse()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gbtopk(args, rank, world, local)
    barrier()


if __name__ == "__main__":
    main()
