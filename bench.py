#!/usr/bin/env python3
"""Benchmark of the batched variable-length exact top-K (DSA indexer top-K).

Headline workload: the DSv3.2-like decode batch - 64 rows x 163840 fp32
logits, seq_lens ~U[2048, 163840], top_k = 2048, previous-step hint given
(seeded synthetic inputs from ``workloads``; the pages' real decode captures
are not available).  One step = one ``gbtopk_varlen`` call over the batch.
The same JSON line carries, under ``workloads``, the other configurations
timed the same way: the decode batch without its hint, the 1024-row
long-row sweep (1024 x 262144 fp32, top_k 2048, hinted), the DSv4-like MTP
batch (512 x 65536 bf16, next_n 4, compress_ratio 4, top_k 1024), the short
rows (4096 x 2048 fp16, top_k 512) and the compact page-table transform
(256 x 32768 fp32 in a 33024-wide buffer, page_size 64, sorted, top_k 2048).

Timing: W untimed warm-up steps, then exactly K steps captured as one CUDA
graph and replayed once, timed with CUDA events on the launching stream and
bracketed by barrier + synchronize; inputs rotate over enough device copies
that the valid bytes touched between two uses of a copy exceed 3x the
129 MB L2 (no flush needed).  ``value`` = rows/s over all ranks (max time
over ranks).  ``e2e`` repeats the headline through the public Python API
with pinned host inputs copied in and indices copied out each step.
``--impl reference`` times the CPU oracle on the host cores (rank 0 only).

Multi-GPU: rows are independent, so each rank runs its own batch (weak
scaling, replicas, no collective on the data path).  ``--gpus N`` without a
launcher starts the N ranks itself through torch.distributed.run.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import socket
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

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
    ("dsv32_decode", "6e3fa146b8453f19"): 21_878_272,   # row 2,365,952 + chunk 19,512,320
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gbtopk", "reference"], default="gbtopk")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dsv32_decode",
                    help="the headline workload (the metric's configuration by default)")
    ap.add_argument("--extra-steps", type=int, default=50,
                    help="timed steps of each of the other workloads")
    ap.add_argument("--no-extra", action="store_true", help="time the headline workload only")
    ap.add_argument("--sweep-rows", type=int, default=1024,
                    help="rows of the long-row sweep (a smaller batch for profiler captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="short run for profilers: warm-up + K eager steps of the headline, "
                         "no clock sampling, no e2e, no CPU leg, no other workloads")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed

def spawn_ranks(n_gpus: int) -> int:
    """Runs this script as n_gpus ranks through torch.distributed.run (when
    it was started without a launcher); returns their exit status."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n_gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def dist_init(n_gpus: int):
    """Returns (rank, world, local_rank); initialises torch.distributed for N>1."""
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"bench.py: --gpus {n_gpus} but WORLD_SIZE={world}")
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


# ------------------------------------------------------------------ workloads

SWEEP_ROWS = [1024]   # --sweep-rows


def _varlen_case(name: str, rank: int):
    import workloads
    s = 17 * rank
    if name == "dsv32_decode":
        return workloads.dsv32_decode(seed=2000 + s)
    if name == "dsv32_decode_nohint":
        return workloads.dsv32_decode(hinted=False, seed=2000 + s)
    if name == "long_row_sweep_1024":
        return workloads.long_row_sweep(SWEEP_ROWS[0], 2048, True, seed=3999 + s)
    if name == "dsv4_mtp":
        return workloads.dsv4_mtp(seed=4000 + s)
    if name == "short_rows":
        return workloads.short_rows(seed=4100 + s)
    raise KeyError(name)


WORKLOADS = {
    "dsv32_decode": "dsv32_decode: 64 rows x 163840 fp32, top_k=2048, seq_lens U[2048,163840], hint=yes",
    "dsv32_decode_nohint": "dsv32_decode: 64 rows x 163840 fp32, top_k=2048, seq_lens U[2048,163840], hint=no",
    "long_row_sweep_1024": "long_row_sweep: 1024 rows x 262144 fp32, top_k=2048, seq_lens U[131072,262144], hint=yes",
    "dsv4_mtp": "dsv4_mtp: 512 rows (128 requests x next_n 4) x 65536 bf16, compress_ratio 4, top_k=1024, "
                "seq_lens U[0,262144] with four requests at 0..3, hint=no",
    "short_rows": "short_rows: 4096 rows x 2048 fp16, top_k=512, seq_lens U[1,2048]",
    "page_table": "page_table: 256 rows x 32768 fp32 in a 33024-wide buffer, ragged row_starts, "
                  "page_size 64, page table 256 x 1024, top_k=2048, out + out_raw, sorted",
}


def varlen_valid_columns(seq_lens, R, W, next_n, cr):
    """Valid columns per row from the public contract (FlashInfer
    `top_k_varlen`, seq_lens): max(0, seq - next_n + t + 1) // cr, at most W."""
    out = []
    for r in range(R):
        num = int(seq_lens[r // next_n]) - next_n + (r % next_n) + 1
        out.append(0 if num <= 0 else min(num // cr, W))
    return out


class Timed:
    """One workload: device input copies, a step, the algorithmic bytes."""

    def __init__(self, name, dev, rank):
        import torch
        import sparse_attention_top_gb300 as gb
        self.name = name
        self.label = WORKLOADS[name]
        self.gb = gb
        if name == "page_table":
            import workloads
            c = workloads.page_table_case(seed=5000 + 17 * rank)
            R, W = c.scores.shape
            S = c.scores.stride(0)
            self.rows, self.top_k, self.dtype = R, c.top_k, c.scores.dtype
            n = [max(0, min(int(c.lengths[r]), W - int(c.row_starts[r]))) for r in range(R)]
            valid = 4 * sum(n)
            self.algo_bytes = valid + R * c.top_k * 8          # columns read + out + out_raw
            full = torch.as_strided(c.scores, (R, S), (S, 1)).contiguous()
            self.copies = max(2, -(-3 * L2_BYTES // max(valid, 1)) + 1)
            self.x = [full.to(dev)[:, :W] for _ in range(self.copies)]
            self.lengths = c.lengths.to(dev)
            self.row_starts = c.row_starts.to(dev)
            self.pt = c.page_table.to(dev)
            self.pt_starts = c.page_table_row_starts.to(dev)
            self.page_size = c.page_size
            self.out = torch.empty(R, c.top_k, dtype=torch.int32, device=dev)
            self.raw = torch.empty(R, c.top_k, dtype=torch.int32, device=dev)
            self.flags = gb.SORTED if c.deterministic else 0
            self.ws = torch.zeros(gb.gbtopk_workspace_bytes(R, W, c.top_k, c.scores.dtype),
                                  dtype=torch.uint8, device=dev)
            self.hinted = False
            self.case = None
            self.width = W
        else:
            c = _varlen_case(name, rank)
            R, W = c.logits.shape
            self.case = c
            self.rows, self.top_k, self.dtype, self.width = R, c.top_k, c.logits.dtype, W
            es = c.logits.element_size()
            n = varlen_valid_columns(c.seq_lens.tolist(), R, W, c.next_n, c.compress_ratio)
            valid = es * sum(n)
            self.algo_bytes = valid + R * c.top_k * 4          # columns read + indices written
            self.copies = max(2, -(-3 * L2_BYTES // max(valid, 1)) + 1)
            self.x = [c.logits.to(dev) for _ in range(self.copies)]
            self.seq = c.seq_lens.to(dev)
            self.hint = [c.pre_idx.to(dev) for _ in range(self.copies)] if c.pre_idx is not None else None
            self.out = torch.empty(R, c.top_k, dtype=torch.int32, device=dev)
            self.flags = 0
            self.ws = torch.zeros(gb.gbtopk_workspace_bytes(R, W, c.top_k, c.logits.dtype),
                                  dtype=torch.uint8, device=dev)
            self.hinted = c.pre_idx is not None
        plan = gb.gbtopk_plan_query(self.rows, self.width, self.top_k, self.dtype)
        if not plan["split"]:
            self.kernels_per_call = 1
            self.path = "one warp per row" if (self.width <= 2048 and not self.flags) else "one block per row"
        elif plan["fused"]:
            self.kernels_per_call = 2
            self.path = "row guess + chunk kernel (finalize in the row's last chunk block)"
        else:
            self.kernels_per_call = 3
            self.path = "row guess + persistent stream kernel + finalize kernel"

    def step(self, i):
        gb = self.gb
        j = i % self.copies
        if self.case is None:
            gb.gbtopk_page_table_transform(self.x[j], self.lengths, self.row_starts, self.pt,
                                           self.pt_starts, self.page_size, self.top_k, self.out,
                                           self.raw, self.flags, self.ws)
        else:
            c = self.case
            gb.gbtopk_varlen(self.x[j], self.seq, self.top_k, self.hint[j] if self.hint else None,
                             c.next_n, c.compress_ratio, self.out, None, self.flags, self.ws)


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


# ------------------------------------------------------------------ oracle legs

def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine() or "unknown"


def oracle_rows_per_s(case, seconds: float, threads: int, rows_per_task: int = 4):
    """The oracle as it stands, on `threads` host threads (each call releases
    the interpreter lock), cycling over the batch's rows for about `seconds`."""
    import oracle
    oracle.build()
    R = case.logits.shape[0]
    nn, cr = case.next_n, case.compress_ratio
    if nn != 1:
        rows_per_task = max(nn, rows_per_task - rows_per_task % nn)

    def task(r0):
        sl = slice(r0, r0 + rows_per_task)
        oracle.topk_varlen(case.logits[sl], case.seq_lens[r0 // nn:(r0 + rows_per_task) // nn],
                           case.top_k, nn, cr, return_values=False)
        return case.logits[sl].shape[0]

    done, r = 0, 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        while time.perf_counter() - t0 < seconds:
            starts = [(r + i * rows_per_task) % R for i in range(threads)]
            starts = [s - s % nn for s in starts]
            done += sum(ex.map(task, starts))
            r = (r + threads * rows_per_task) % R
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def run_reference(args, rank, world):
    if rank != 0:
        return
    case = _varlen_case(args.workload, 0) if args.workload != "page_table" else None
    if case is None:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the varlen "
                          "oracle; choose a varlen workload"}), flush=True)
        return
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    R, W = case.logits.shape
    rows_per_task = 4
    r = 0

    def task(r0):
        oracle.topk_varlen(case.logits[r0:r0 + rows_per_task], case.seq_lens[r0:r0 + rows_per_task],
                           case.top_k, return_values=False)

    ex = ThreadPoolExecutor(threads)

    def step():
        nonlocal r
        list(ex.map(task, [(r + i * rows_per_task) % R for i in range(threads)]))
        r = (r + threads * rows_per_task) % R

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    ex.shutdown()
    rows = threads * rows_per_task * args.steps
    v = rows / dt
    sample = (f"{threads * rows_per_task} rows of the {args.workload} batch per step "
              f"({R} rows x {W}, k={case.top_k}), {threads} host threads ({cpu_model()})")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOADS[args.workload]},
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg

def time_graph(w: Timed, steps: int, warmup: int, dev, sampler=None):
    """Warm-up eager steps, then `steps` steps captured in one CUDA graph and
    replayed once; returns (ms for the K steps, eager ms for K steps, clocks)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    for i in range(max(warmup, 3)):
        w.step(i)
    torch.cuda.synchronize(dev)
    gstream = torch.cuda.Stream(dev)
    gstream.wait_stream(stream)
    with torch.cuda.stream(gstream):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gstream):
            for s_ in range(steps):
                w.step(s_)
    torch.cuda.synchronize(dev)

    def timed(run):
        barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        run()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return t0.elapsed_time(t1)

    clocks = None
    if sampler is not None:
        # keep the GPU busy ~1 s around the timed region so the clock samples
        # reflect it (the untimed replays also serve as warm-up)
        with sampler as clk:
            t_end = time.perf_counter() + 0.6
            while time.perf_counter() < t_end:
                graph.replay()
            torch.cuda.synchronize(dev)
            total_ms = timed(graph.replay)
            t_end = time.perf_counter() + 0.4
            while time.perf_counter() < t_end:
                graph.replay()
            torch.cuda.synchronize(dev)
        clocks = clk.summary()
    else:
        graph.replay()
        torch.cuda.synchronize(dev)
        total_ms = timed(graph.replay)
    eager_ms = timed(lambda: [w.step(s_) for s_ in range(steps)])
    del graph
    return total_ms, eager_ms, clocks


def run_gbtopk(args, rank, world, local):
    import torch
    import sparse_attention_top_gb300 as gb

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    head = Timed(args.workload, dev, rank)
    if args.profile:
        for i in range(max(args.warmup, 3)):
            head.step(i)
        torch.cuda.synchronize(dev)
        for s in range(args.steps):
            head.step(s)
        torch.cuda.synchronize(dev)
        if rank == 0:
            print(json.dumps({"profile_run": True, "workload": args.workload, "steps": args.steps,
                              "rows": head.rows, "width": head.width,
                              "algorithmic_bytes_per_launch": head.algo_bytes}), flush=True)
        return

    peak, peak_src = peak_hbm()
    total_ms, eager_ms, clocks = time_graph(head, args.steps, args.warmup, dev, ClockSampler(local))
    total_ms_max = reduce_max(total_ms)
    eager_ms_max = reduce_max(eager_ms)
    rows_all = reduce_sum(head.rows * args.steps)
    value = rows_all / (total_ms_max / 1e3)
    avg_launch_s = total_ms / args.steps / 1e3
    achieved = head.algo_bytes / avg_launch_s / 1e9
    traffic = NCU_TRAFFIC.get((args.workload, kernel_sha()))

    extra = {}
    if not args.no_extra and world == 1:
        for name in WORKLOADS:
            if name == args.workload:
                continue
            w = Timed(name, dev, rank)
            ms, ems, _ = time_graph(w, args.extra_steps, max(3, min(args.warmup, 10)), dev)
            us = ms / args.extra_steps * 1e3
            gbs = w.algo_bytes / (us * 1e-6) / 1e9
            extra[name] = {"workload": w.label, "path": w.path, "steps": args.extra_steps,
                           "ms_per_step": ms / args.extra_steps, "us_per_call": us,
                           "rows_per_s": w.rows / (us * 1e-6), "algorithmic_bytes": w.algo_bytes,
                           "achieved_gbs": gbs, "frac": gbs / peak,
                           "eager_us_per_call": ems / args.extra_steps * 1e3,
                           "kernels_per_call": w.kernels_per_call,
                           "l2": f"inputs rotate over {w.copies} device copies"}
            del w
            torch.cuda.empty_cache()

    e2e = None
    if not args.no_e2e and head.case is not None:
        e2e = run_e2e(head.case, dev, args, gb)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and head.case is not None:
        threads = os.cpu_count() or 1
        v1, rows1, secs1 = oracle_rows_per_s(head.case, 8.0, 1)
        vn, rowsn, secsn = oracle_rows_per_s(head.case, 8.0, threads)
        cpu = {"value": vn, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{rowsn} rows of this batch on {threads} host threads "
                         f"(4 rows per task, cycling), {secsn:.1f} s",
               "single_thread": {"value": v1, "unit": "rows/s", "cores": 1,
                                 "sample": f"{rows1} rows, {secs1:.1f} s"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[head.dtype],
            "data": "synthetic",
            "config": {"workload": head.label, "rows": head.rows, "width": head.width,
                       "top_k": head.top_k, "hinted": head.hinted,
                       "l2": f"inputs rotate over {head.copies} device copies "
                             f"(valid bytes between two uses of a copy > 3x L2)",
                       "parallelism": f"replicas x{world} (rows independent)"},
            "gpu_launches": args.steps * head.kernels_per_call,
            "timing": {"mode": "one CUDA graph of the K steps, replayed once",
                       "kernels_per_call": head.kernels_per_call, "path": head.path,
                       "eager_ms_per_step": eager_ms_max / args.steps},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": head.algo_bytes,
                         "avg_launch_us": avg_launch_s * 1e6,
                         "kernel": f"the whole call ({head.path})"},
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "workloads": extra,
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
        gb.top_k_varlen(d_logits, d_seq, k, pre_idx=d_hint, compress_ratio=case.compress_ratio,
                        next_n=case.next_n, out_indices=d_out)
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
    h2d = (h_logits.numel() * h_logits.element_size() + h_seq.numel() * 4
           + (h_hint.numel() * 4 if h_hint is not None else 0))
    return {"value": rows / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": R * k * 4, "steps": steps}


def main():
    args = parse()
    SWEEP_ROWS[0] = args.sweep_rows
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args.gpus))
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gbtopk(args, rank, world, local)
    barrier()


if __name__ == "__main__":
    main()
