"""Benchmark: single-query paged-attention decode on GB300.

Metric: paged decode us/call and KV-read GB/s (fraction of GB300 HBM peak) vs
context. The headline `value` is the whole-job KV-read throughput (GB/s) of one
step; the per-call curve (us/call and GB/s per cell) rides along in `curve`.

Default workload (N=1): the GQA x depth grid of "vLLM's custom ROCm
paged-attention kernel wins all sixty cells" (§1, Figure 1): head_dim 128,
block 16, bf16 N(0,1); (Hq, Hkv) in (8,8) (16,8) (24,8) (32,8) (32,16); seq_len
1K..32K; batch 1 and 8; randomly permuted block tables over a pool twice the
used blocks with zero-filled spare. A step runs every one of the 60 cells once,
each on its own resident cache (about 13 GiB of distinct KV per step, so no cell
is read from L2 by a later visit). The step is captured once in a CUDA graph and
replayed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload grid|hybrid|mixed|first]

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (there is no other implementation to run). With torchrun (N > 1) every
rank runs an independent replica (the decode path has no exchange step) and
value = bytes of all ranks / max over ranks of the step time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode µs/call and KV-read GB/s (fraction of GB300 HBM peak) "
          "vs context")
GRID_SHAPES = [(8, 8), (16, 8), (24, 8), (32, 8), (32, 16)]
GRID_LENS = [1024, 2048, 4096, 8192, 16384, 32768]
GRID_BATCHES = [1, 8]
HYBRID_LENS = [500, 1024, 2048, 4096, 8192, 12288, 16384, 20480, 24576, 28672, 32768]
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------- workloads
class Cell:
    """One decode call with its inputs resident on the device."""

    def __init__(self, B, Hq, Hkv, D, bs, lens, seed, device, poison=None, pool_factor=2.0,
                 tag=""):
        self.B, self.Hq, self.Hkv, self.D, self.bs = B, Hq, Hkv, D, bs
        self.lens = list(lens)
        self.tag = tag
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        nblk = [-(-L // bs) for L in lens]
        used = sum(nblk)
        nb = max(1, int(math.ceil(used * pool_factor)))
        self.num_blocks = nb
        dt = torch.bfloat16
        self.q = torch.randn((B, Hq, D), generator=gen, device=device).to(dt)
        fill = float("nan") if poison == "nan" else 0.0
        self.k = torch.full((nb, bs, Hkv, D), fill, dtype=dt, device=device)
        self.v = torch.full((nb, bs, Hkv, D), fill, dtype=dt, device=device)
        perm = torch.randperm(nb, generator=gen, device=device)
        mb = max(nblk)
        bt = torch.full((B, mb), -1, dtype=torch.int32, device=device)
        off = 0
        for b, L in enumerate(lens):
            n = nblk[b]
            bt[b, :n] = perm[off:off + n].to(torch.int32)
            off += n
            # live tokens get N(0,1); the unwritten tail of the last block keeps the fill
            t = torch.arange(L, device=device)
            phys = bt[b, (t // bs)].long()
            slot = t % bs
            self.k[phys, slot] = torch.randn((L, Hkv, D), generator=gen, device=device).to(dt)
            self.v[phys, slot] = torch.randn((L, Hkv, D), generator=gen, device=device).to(dt)
        self.bt = bt
        self.sl = torch.tensor(lens, dtype=torch.int32, device=device)
        self.out = torch.empty_like(self.q)
        self.max_len = max(lens)
        self.scale = float(np.float32(1.0 / math.sqrt(D)))
        self.ws = None

    def kv_bytes(self) -> int:
        return sum(self.lens) * self.Hkv * self.D * 2 * 2

    def alg_bytes(self) -> int:
        """Bytes the method must move: KV, the live block-table entries, q, out, seq_lens."""
        table = sum(-(-L // self.bs) for L in self.lens) * 4
        return self.kv_bytes() + table + 2 * self.B * self.Hq * self.D * 2 + 4 * self.B

    def call(self, pa, stream=None):
        pa.decode(self.q, self.k, self.v, self.bt, self.sl, self.scale, out=self.out,
                  max_seq_len=self.max_len, workspace=self.ws, stream=stream)


def build_workload(name, device, seed=0):
    cells = []
    if name == "grid":
        i = 0
        for B in GRID_BATCHES:
            for hq, hkv in GRID_SHAPES:
                for L in GRID_LENS:
                    cells.append(Cell(B, hq, hkv, 128, 16, [L] * B, seed + i, device,
                                      tag=f"{hq}/{hkv} B={B} L={L}"))
                    i += 1
        desc = {"workload": "gqa_depth_grid", "head_dim": 128, "block_size": 16,
                "shapes_hq_hkv": GRID_SHAPES, "seq_lens": GRID_LENS, "batches": GRID_BATCHES,
                "cells": len(cells), "pool": "2x used blocks, zero-filled spare"}
    elif name == "hybrid":
        # 16 independent layer caches per context length: 24q/4kv, head 256, block 784
        i = 0
        for L in HYBRID_LENS:
            for layer in range(16):
                cells.append(Cell(1, 24, 4, 256, 784, [L], seed + i, device,
                                  tag=f"hybrid L={L} layer={layer}"))
                i += 1
        desc = {"workload": "hybrid_full_attention_layer", "Hq": 24, "Hkv": 4, "head_dim": 256,
                "block_size": 784, "batch": 1, "seq_lens": HYBRID_LENS, "layers_per_step": 16,
                "cells": len(cells)}
    elif name == "mixed":
        import pa_inputs as pi
        lens = pi.uniform_seq_lens(64, 1024, 32768, seed=seed)
        cells.append(Cell(64, 32, 8, 128, 16, lens, seed, device, poison="nan",
                          pool_factor=1.1, tag="mixed B=64"))
        desc = {"workload": "mixed_serving_batch", "batch": 64, "Hq": 32, "Hkv": 8,
                "head_dim": 128, "block_size": 16, "seq_lens": "U[1024,32768] seed 0",
                "pool": "shared, 1.1x used blocks, NaN in unwritten slots"}
    elif name == "first":
        cells.append(Cell(1, 8, 8, 128, 16, [512], seed, device, tag="first"))
        desc = {"workload": "first_config", "batch": 1, "Hq": 8, "Hkv": 8, "head_dim": 128,
                "block_size": 16, "seq_len": 512}
    else:
        raise SystemExit(f"unknown workload {name}")
    return cells, desc


# ---------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def timing_event():
    try:
        return torch.cuda.Event(enable_timing=True, external=True), True
    except TypeError:
        return torch.cuda.Event(enable_timing=True), False


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def oracle_sample(budget_s, shapes=GRID_SHAPES, lens=GRID_LENS, D=128, device="cuda"):
    """Time the float64 oracle on B=1 grid cells (contiguous K/V on the host), up to
    about budget_s seconds of oracle time. Returns (bytes, seconds, description)."""
    from oracle import decode_ref
    done_bytes, spent, cells = 0, 0.0, []
    gen = torch.Generator(device=device)
    gen.manual_seed(1234)
    for L in lens:
        for hq, hkv in shapes:
            if spent >= budget_s:
                break
            q = torch.randn((1, hq, D), generator=gen, device=device).to(torch.bfloat16)
            K = torch.randn((L, hkv, D), generator=gen, device=device).to(torch.bfloat16)
            V = torch.randn((L, hkv, D), generator=gen, device=device).to(torch.bfloat16)
            qn = q.double().cpu().numpy()
            Kn = K.double().cpu().numpy()
            Vn = V.double().cpu().numpy()
            t0 = time.perf_counter()
            decode_ref(qn, [Kn], [Vn], 1.0 / math.sqrt(D))
            spent += time.perf_counter() - t0
            done_bytes += L * hkv * D * 2 * 2
            cells.append(f"{hq}/{hkv}@{L}")
    return done_bytes, spent, "float64 oracle, batch-1 grid cells " + ",".join(cells)


# ---------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The float64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    # a step: the five grid shapes at batch 1, seq_len 4096 (bounded sample)
    steps, warm = args.steps, args.warmup
    per_step = []
    total_bytes = 0
    for i in range(warm + steps):
        b, s, desc = oracle_sample(1e9, lens=[4096], device="cuda" if torch.cuda.is_available() else "cpu")
        if i >= warm:
            per_step.append(s)
            total_bytes += b
    secs = sum(per_step)
    gbs = total_bytes / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * secs / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "gqa_depth_grid", "sample": "batch-1 cells of the 5 shapes at "
                   "seq_len 4096 per step", "head_dim": 128, "block_size": 16},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import paged_kv_attention_pa_gb300 as pa
    from paged_kv_attention_pa_gb300 import build as pa_build
    pa_build.build()
    pa.load()

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cells, desc = build_workload(args.workload, dev, seed=args.seed + 1000 * rank)
    stream = torch.cuda.Stream(dev)
    # one workspace per cell so the captured graph has fixed addresses
    for c in cells:
        a = pa.make_args(c.q, c.k, c.v, c.bt, c.sl, c.out, c.scale, c.max_len)
        nbytes = pa.load().pa_decode_ex_workspace_bytes(__import__("ctypes").byref(a))
        c.ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def step_eager():
        for c in cells:
            c.call(pa, stream)

    # warm-up (also loads modules and sets the shared-memory opt-in)
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step_eager()
    stream.synchronize()
    for c in cells:
        assert torch.isfinite(c.out).all(), f"non-finite output in {c.tag}"
        assert pa.read_device_errors(c.ws, stream) == 0, f"device error in {c.tag}"

    # graph A: the step as launched in production (no instrumentation)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step_eager()
    # graph B: the same step with an event pair around every launch (per-launch times)
    ev_pairs = []
    ext_ok = True
    for c in cells:
        e0, ok0 = timing_event()
        e1, ok1 = timing_event()
        ext_ok = ext_ok and ok0 and ok1
        ev_pairs.append((e0, e1))
    graph_b = None
    if ext_ok:
        graph_b = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph_b, stream=stream):
                for c, (e0, e1) in zip(cells, ev_pairs):
                    e0.record(stream)
                    c.call(pa, stream)
                    e1.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()

    # ---------------- timed region: K graph replays
    clocks = ClockSampler(dev.index) if rank == 0 else None
    if clocks:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = starts[0].elapsed_time(ends[-1])

    # ---------------- per-launch durations (graph B, or eager with events)
    per_launch = [[] for _ in cells]
    reps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        for _ in range(reps):
            if graph_b is not None:
                graph_b.replay()
            else:
                for c, (e0, e1) in zip(cells, ev_pairs):
                    e0.record(stream)
                    c.call(pa, stream)
                    e1.record(stream)
            stream.synchronize()
            for i, (e0, e1) in enumerate(ev_pairs):
                per_launch[i].append(e0.elapsed_time(e1))
    if clocks:
        clk = clocks.stop()
    else:
        clk = None

    # ---------------- end to end through the public API with host buffers
    host_q = [torch.empty(c.q.shape, dtype=c.q.dtype, pin_memory=True) for c in cells]
    host_bt = [torch.empty(c.bt.shape, dtype=c.bt.dtype, pin_memory=True) for c in cells]
    host_sl = [torch.empty(c.sl.shape, dtype=c.sl.dtype, pin_memory=True) for c in cells]
    host_out = [torch.empty(c.out.shape, dtype=c.out.dtype, pin_memory=True) for c in cells]
    for c, hq, hb, hs in zip(cells, host_q, host_bt, host_sl):
        hq.copy_(c.q)
        hb.copy_(c.bt)
        hs.copy_(c.sl)
    h2d = sum(t.numel() * t.element_size() for t in host_q + host_bt + host_sl)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def step_e2e():
        for c, hq, hb, hs, ho in zip(cells, host_q, host_bt, host_sl, host_out):
            c.q.copy_(hq, non_blocking=True)
            c.bt.copy_(hb, non_blocking=True)
            c.sl.copy_(hs, non_blocking=True)
            c.call(pa, stream)
            ho.copy_(c.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_e2e()
    stream.synchronize()
    e2e_steps = max(3, args.steps)
    es = torch.cuda.Event(enable_timing=True)
    ee = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        es.record(stream)
        for _ in range(e2e_steps):
            step_e2e()
        ee.record(stream)
    stream.synchronize()
    e2e_ms = es.elapsed_time(ee) / e2e_steps

    # ---------------- aggregate over ranks
    kv = sum(c.kv_bytes() for c in cells)
    alg = sum(c.alg_bytes() for c in cells)
    ms_step = total_ms / args.steps
    t = torch.tensor([ms_step, e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_step_max, e2e_max = float(t[0]), float(t[1])
    value = world * kv / (ms_step_max * 1e-3) / 1e9
    e2e_value = world * kv / (e2e_max * 1e-3) / 1e9
    if rank != 0:
        return

    peak, peak_kind = load_peaks()
    launch_ms = [statistics.median(x) for x in per_launch]
    kernel_ms_total = sum(launch_ms)
    achieved = alg / (kernel_ms_total * 1e-3) / 1e9
    curve = []
    for c, ms in zip(cells, launch_ms):
        gbs = c.kv_bytes() / (ms * 1e-3) / 1e9
        curve.append({"cell": c.tag, "us_per_call": round(ms * 1e3, 3),
                      "kv_gbs": round(gbs, 1), "frac": round(gbs / peak, 4)})
    budget = float(os.environ.get("PA_BENCH_CPU_BUDGET_S", "12"))
    cb_bytes, cb_s, cb_desc = oracle_sample(budget, device=dev)
    S, P = pa.plan(cells[-1].B, cells[-1].Hq, cells[-1].Hkv, cells[-1].D, cells[-1].bs,
                   cells[-1].max_len)
    line = {
        "impl": "ours", "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(desc, **{
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "inputs larger than L2: each step reads every cell's own cache once "
                  f"({kv / 2**30:.2f} GiB of distinct KV per step)",
            "timed": "CUDA graph of the whole step, replayed K times, CUDA events",
            "kv_bytes_per_step": kv}),
        "gpu_launches": len(cells) * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_kind": peak_kind, "kernel": "pa::decode_kernel",
                     "alg_bytes_per_launch": alg / len(cells),
                     "avg_launch_us": round(1e3 * kernel_ms_total / len(cells), 3),
                     "launch_timing": "graph with external events" if graph_b is not None
                     else "eager launches with events"},
        "cpu_baseline": {"value": round(cb_bytes / cb_s / 1e9, 4), "unit": "GB/s",
                         "cores": cpu_threads(), "kind": "oracle", "sample": cb_desc},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "what": "per cell: pinned H2D of q, block table, seq_lens; pa.decode; "
                        "D2H of out (KV cache resident)"},
        "clocks": clk,
        "step_ms_min_med_max": [round(min(step_ms), 4), round(statistics.median(step_ms), 4),
                                round(max(step_ms), 4)],
        "plan_last_cell": {"splits": S, "partition_tokens": P},
        "curve": curve,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="grid", choices=["grid", "hybrid", "mixed", "first"])
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
