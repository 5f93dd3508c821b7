"""Benchmark: single-query paged-attention decode on GB300.

Metric: paged decode us/call and KV-read GB/s (fraction of GB300 HBM peak) vs
context. The headline `value` is the whole-job KV-read throughput (GB/s) of one
step; the per-call curve (us/call, GB/s and fraction per cell) rides along in
`curve`.

Default workload (N=1): the GQA x depth grid of "vLLM's custom ROCm
paged-attention kernel wins all sixty cells" (§1, Figure 1): head_dim 128,
block 16, bf16 N(0,1); (Hq, Hkv) in (8,8) (16,8) (24,8) (32,8) (32,16); seq_len
1K..32K; batch 1 and 8; randomly permuted block tables over a pool twice the
used blocks with zero-filled spare. A step runs every one of the 60 cells once,
each on its own resident cache (about 13 GiB of distinct KV per step, so no cell
is read from L2 by a later visit). The step is captured once in a CUDA graph and
replayed K times.

The curve times each cell in steady state: a CUDA graph of back-to-back calls
rotating over enough independent copies of the cell (>= 512 MiB of KV in total,
four times the L2) that every call reads HBM, as an engine replays its layers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload grid|hybrid|mixed|first|cell|window|rows]
                    [--cell Hq,Hkv,B,L,D,bs] [--kv-dtype bf16|fp8] [--no-curve]

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
import re
import statistics
import subprocess
import tempfile
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
ROTATE_BYTES = 512 << 20  # KV per rotation of the steady-state curve (4x the 129 MB L2)
FP8_SCALE = 8.0 / 448.0   # per-tensor scale of the fp8 caches (N(0,1) to 8 sigma)
KV_FP8 = False            # set by --kv-dtype fp8


# ---------------------------------------------------------------------- workloads
class Inst:
    """One set of device inputs for a decode call."""

    def __init__(self, B, Hq, Hkv, D, bs, lens, seed, device, poison, pool_factor, exact,
                 window=0, fp8=False, rows=1):
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        dt = torch.bfloat16
        cdt = torch.float8_e4m3fn if fp8 else dt
        # fp8 caches: stored value = N(0,1) draw / FP8_SCALE (rounded to e4m3)
        cv = (lambda x: (x.float() / FP8_SCALE).to(cdt)) if fp8 else (lambda x: x.to(dt))
        nblk = [-(-L // bs) for L in lens]
        # timing copies of a windowed call back only the blocks the window can touch;
        # earlier logical blocks share them (they are never read)
        back = [min(n, -(-window // bs) + 1) if (window > 0 and not exact) else n for n in nblk]
        nb = max(1, int(math.ceil(sum(back) * pool_factor)))
        self.num_blocks = nb
        qshape = (B, rows, Hq, D) if rows > 1 else (B, Hq, D)
        self.q = torch.randn(qshape, generator=gen, device=device).to(dt)
        if exact:
            # live tokens N(0,1); spare blocks and unwritten tails keep the fill
            fill = float("nan") if poison == "nan" else 0.0
            self.k = torch.full((nb, bs, Hkv, D), fill, dtype=cdt, device=device)
            self.v = torch.full((nb, bs, Hkv, D), fill, dtype=cdt, device=device)
        else:
            # timing copies: the whole pool N(0,1) (values do not change the work)
            self.k = cv(torch.randn((nb, bs, Hkv, D), generator=gen, device=device))
            self.v = cv(torch.randn((nb, bs, Hkv, D), generator=gen, device=device))
        perm = torch.randperm(nb, generator=gen, device=device)
        bt = torch.full((B, max(nblk)), -1, dtype=torch.int32, device=device)
        off = 0
        for b, L in enumerate(lens):
            n, m = nblk[b], back[b]
            own = perm[off:off + m].to(torch.int32)
            # the last m logical blocks get their own physical blocks, in order
            bt[b, n - m:n] = own
            if n > m:
                bt[b, :n - m] = own[torch.arange(n - m, device=device) % m]
            off += m
            if exact:
                t = torch.arange(L, device=device)
                phys = bt[b, (t // bs)].long()
                self.k[phys, t % bs] = cv(torch.randn((L, Hkv, D), generator=gen, device=device))
                self.v[phys, t % bs] = cv(torch.randn((L, Hkv, D), generator=gen, device=device))
        self.bt = bt
        self.sl = torch.tensor(lens, dtype=torch.int32, device=device)
        self.out = torch.empty_like(self.q)


class Cell:
    """A decode configuration: inputs for the step, plus copies for the curve."""

    def __init__(self, B, Hq, Hkv, D, bs, lens, seed, device, poison=None, pool_factor=2.0,
                 tag="", window=0, fp8=None, rows=1):
        self.B, self.Hq, self.Hkv, self.D, self.bs = B, Hq, Hkv, D, bs
        self.rows = rows
        self.window = window
        self.fp8 = KV_FP8 if fp8 is None else fp8
        self.kv_elem = 1 if self.fp8 else 2
        self.lens = list(lens)
        self.tag = tag
        self.seed, self.device, self.poison, self.pool_factor = seed, device, poison, pool_factor
        self.insts = [Inst(B, Hq, Hkv, D, bs, lens, seed, device, poison, pool_factor, True,
                           window, self.fp8, rows)]
        self.max_len = max(lens)
        self.total_tokens = sum(self.lens)  # host-side planning hint, like max_len
        self.scale = float(np.float32(1.0 / math.sqrt(D)))
        self.ws = None

    def add_copies(self, n):
        for i in range(len(self.insts), n):
            self.insts.append(Inst(self.B, self.Hq, self.Hkv, self.D, self.bs, self.lens,
                                   self.seed + 7919 * i, self.device, self.poison,
                                   self.pool_factor, False, self.window, self.fp8, self.rows))

    def read_lens(self):
        """Tokens each sequence's query attends to (the window bounds them)."""
        return [min(L, self.window) if self.window > 0 else L for L in self.lens]

    def kv_bytes(self) -> int:
        return sum(self.read_lens()) * self.Hkv * self.D * 2 * self.kv_elem

    def alg_bytes(self) -> int:
        """Bytes the method must move: KV, the live block-table entries, q, out, seq_lens."""
        table = sum(-(-L // self.bs) + 1 for L in self.read_lens()) * 4
        return self.kv_bytes() + table + 2 * self.B * self.rows * self.Hq * self.D * 2 + 4 * self.B

    def call(self, pa, stream=None, i=0):
        x = self.insts[i]
        self.call_with(pa, stream, x.q, x.bt, x.sl, x.out, i)

    def call_with(self, pa, stream, q, bt, sl, out, i=0):
        """The decode call on copy i's caches with the given q, table, lengths, out."""
        x = self.insts[i]
        pa.decode(q, x.k, x.v, bt, sl, self.scale, out=out, max_seq_len=self.max_len,
                  workspace=self.ws, stream=stream, window=self.window,
                  k_scale=FP8_SCALE, v_scale=FP8_SCALE, total_tokens=self.total_tokens)


def parse_cell(spec):
    hq, hkv, B, L, D, bs = (int(x) for x in spec.split(","))
    return hq, hkv, B, L, D, bs


def build_workload(name, device, seed=0, cell_spec=None, fp8=None, lens=None):
    """The cells of a workload. fp8 overrides --kv-dtype for these cells (their tags
    then start with 'fp8 '); lens restricts the hybrid layer's context lengths."""
    cells = []
    pre = "fp8 " if fp8 else ""
    if name == "grid":
        i = 0
        for B in GRID_BATCHES:
            for hq, hkv in GRID_SHAPES:
                for L in GRID_LENS:
                    cells.append(Cell(B, hq, hkv, 128, 16, [L] * B, seed + i, device,
                                      tag=f"{pre}{hq}/{hkv} B={B} L={L}", fp8=fp8))
                    i += 1
        desc = {"workload": "gqa_depth_grid", "head_dim": 128, "block_size": 16,
                "shapes_hq_hkv": GRID_SHAPES, "seq_lens": GRID_LENS, "batches": GRID_BATCHES,
                "cells": len(cells), "pool": "2x used blocks, zero-filled spare"}
    elif name == "hybrid":
        # 16 independent layer caches per context length: 24q/4kv, head 256, block 784
        i = 0
        for L in (lens or HYBRID_LENS):
            for layer in range(16):
                cells.append(Cell(1, 24, 4, 256, 784, [L], seed + i, device,
                                  tag=f"{pre}hybrid L={L} layer={layer}", fp8=fp8))
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
    elif name == "window":
        # sliding-window layers: 32 query / 16 KV heads, head 128, block 16, W = 1024
        i = 0
        for B in GRID_BATCHES:
            for L in GRID_LENS:
                cells.append(Cell(B, 32, 16, 128, 16, [L] * B, seed + i, device,
                                  tag=f"window 32/16 B={B} L={L}", window=1024))
                i += 1
        desc = {"workload": "sliding_window_layer", "Hq": 32, "Hkv": 16, "head_dim": 128,
                "block_size": 16, "window": 1024, "seq_lens": GRID_LENS,
                "batches": GRID_BATCHES, "cells": len(cells),
                "bytes": "KV of the window only: min(L, 1024) tokens per sequence"}
    elif name == "rows":
        # speculative decode: 4 query rows per sequence, 32 query / 8 KV heads, head 128
        i = 0
        for B in GRID_BATCHES:
            for L in GRID_LENS:
                cells.append(Cell(B, 32, 8, 128, 16, [L] * B, seed + i, device,
                                  tag=f"rows4 32/8 B={B} L={L}", rows=4))
                i += 1
        desc = {"workload": "speculative_decode_rows", "Hq": 32, "Hkv": 8, "head_dim": 128,
                "block_size": 16, "query_rows": 4, "seq_lens": GRID_LENS,
                "batches": GRID_BATCHES, "cells": len(cells),
                "bytes": "KV read once per (sequence, KV head) for all 4 rows"}
    elif name == "first":
        cells.append(Cell(1, 8, 8, 128, 16, [512], seed, device, tag="first"))
        desc = {"workload": "first_config", "batch": 1, "Hq": 8, "Hkv": 8, "head_dim": 128,
                "block_size": 16, "seq_len": 512}
    elif name == "cell":
        hq, hkv, B, L, D, bs = parse_cell(cell_spec or "32,8,8,16384,128,16")
        cells.append(Cell(B, hq, hkv, D, bs, [L] * B, seed, device,
                          tag=f"{hq}/{hkv} B={B} L={L} D={D} bs={bs}"))
        desc = {"workload": "single_cell", "Hq": hq, "Hkv": hkv, "batch": B, "seq_len": L,
                "head_dim": D, "block_size": bs}
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


# DRAM traffic of decode_kernel per algorithmic KV byte, from ncu captures of single
# cells (dram__bytes_read.sum + dram__bytes_write.sum, mean over the captured
# launches), keyed by (head_dim, KV type) and scaled to a call by its KV bytes.
# A capture holds only for the kernel code it was taken on: when the SHA-256 of that
# code (comments and blank space removed) differs from the one recorded here, the
# bench reports traffic as null.
TRAFFIC_SOURCES_SHA256 = "0778e44d82c1a835ccc56a9cc2632d31190f3d498e76eb71bc8b29a9b3c31eb4"
TRAFFIC_CAPTURES = {
    # 32q/8kv, block 16, batch 8, 16384 tokens: three launches
    (128, "bf16"): {"alg_bytes": 536870912, "dram_bytes": 537046101 + 1096960},
    # 24q/4kv, block 784, batch 1, 32768 tokens: three launches
    (256, "bf16"): {"alg_bytes": 134217728, "dram_bytes": 134300245 + 1057621},
    # 32q/8kv fp8 E4M3 KV, block 16, batch 8, 16384 tokens: three launches
    (128, "fp8"): {"alg_bytes": 268435456, "dram_bytes": 268605269 + 975360},
}


def code_tokens(src: str) -> str:
    """C/C++/CUDA source with comments and blank space removed: what the compiler
    sees of it, so that edits to comments leave a fingerprint unchanged."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_sources_sha256(csrc=None) -> str:
    """SHA-256 of the device code (comments and blank space removed): the kernel
    headers, the launch parameters and the instantiation units (host-side planning
    and the C API are not part of it)."""
    import hashlib
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "paged_kv_attention_pa_gb300", "csrc")
    files = sorted(f for f in os.listdir(csrc)
                   if f.endswith(".cuh") or f == "pa_params.h" or f.startswith("pa_inst_"))
    for f in files:
        h.update(f.encode())
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()


def traffic_per_call(alg_bytes_per_call: float, D: int, kv: str):
    """(bytes, note): DRAM bytes of one decode call scaled from the matching capture,
    or (None, why)."""
    cap = TRAFFIC_CAPTURES.get((D, kv))
    if cap is None:
        return None, f"no ncu capture for head_dim {D}, {kv} KV"
    if kernel_sources_sha256() != TRAFFIC_SOURCES_SHA256:
        return None, "kernel sources changed since the ncu capture"
    ratio = cap["dram_bytes"] / cap["alg_bytes"]
    return round(alg_bytes_per_call * ratio), (
        f"ncu dram bytes / algorithmic bytes = {ratio:.5f} on a head_dim {D} {kv} cell, "
        "scaled by the call's KV bytes")


def hybrid_linearity(curve, min_tokens=4096):
    """Least-squares fit of µs/call against context for the hybrid layer's cells
    (batch 1, 4 KV heads) of at least min_tokens, with its R^2; None without 3 points."""
    pts = []
    for c in curve:
        m = re.match(r"hybrid L=(\d+)$", c["cell"])
        if m and int(m.group(1)) >= min_tokens:
            pts.append((int(m.group(1)), float(c["us_per_call"])))
    if len(pts) < 3:
        return None
    x = np.array([p[0] / 1024.0 for p in pts])
    y = np.array([p[1] for p in pts])
    A = np.vstack([x, np.ones_like(x)]).T
    (slope, icpt), *_ = np.linalg.lstsq(A, y, rcond=None)
    ss_tot = float(((y - y.mean()) ** 2).sum())
    r2 = 1.0 - float(((y - A @ np.array([slope, icpt])) ** 2).sum()) / ss_tot if ss_tot > 0 else 1.0
    return {"range_tokens": [min(p[0] for p in pts), max(p[0] for p in pts)],
            "slope_us_per_1k_tokens": round(float(slope), 4),
            "intercept_us": round(float(icpt), 3), "r2": round(r2, 5)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the raw samples: PA_BENCH_CLOCKS_DIR if set, else the system's temporary folder
        out_dir = os.environ.get("PA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"pa_bench_clocks_gpu{index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
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
        with open(self.path) as f:
            lines = f.readlines()
        if not os.environ.get("PA_BENCH_CLOCKS_DIR"):
            os.remove(self.path)  # a temporary file unless the caller asked to keep it
        for line in lines:
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


class NvmlSampler:
    """SM clock and clock-event reasons of one GPU, read through NVML (ctypes, read-only
    queries) every ~2 ms on a background thread, so that a timed region of a few tens
    of milliseconds still holds many samples. start() returns False where NVML cannot
    be loaded; the caller then falls back to nvidia-smi."""
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}
    NVML_CLOCK_SM = 1

    def __init__(self, device, period_s=0.002):
        self.device, self.period = device, period_s
        self.samples, self.reasons = [], 0
        self.max_mhz = None
        self.thread, self.stop_flag = None, False

    def _handle(self, lib):
        import ctypes
        h = ctypes.c_void_p()
        try:
            pr = torch.cuda.get_device_properties(self.device)
            bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0:
                return h
        except Exception:
            pass
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device.index or 0), ctypes.byref(h)) == 0:
            return h
        return None

    def start(self):
        import ctypes
        import threading
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = self._handle(lib)
            if h is None:
                return False
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint(0)
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
        except Exception:
            return False

        def loop():
            mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
            while not self.stop_flag:
                if lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) == 0:
                    self.samples.append(float(mhz.value))
                if reasons_fn(h, ctypes.byref(rs)) == 0:
                    self.reasons |= int(rs.value)
                time.sleep(self.period)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()
        return True

    def stop(self):
        if self.thread is None:
            return None
        self.stop_flag = True
        self.thread.join(timeout=5)
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for n, bit in self.REASON_BITS.items() if self.reasons & bit),
                "samples": len(self.samples), "source": "nvml every ~2 ms"}


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


def aggregate_over_ranks(kv_bytes_per_rank, ms_step, e2e_ms, world, device):
    """Whole-job values of a replicas run: every rank processed kv_bytes_per_rank per
    step; the job's step time is the slowest rank's. Returns (value GB/s, e2e GB/s,
    max step ms, max e2e ms)."""
    t = torch.tensor([ms_step, e2e_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_max, e2e_max = float(t[0]), float(t[1])
    value = world * kv_bytes_per_rank / (ms_max * 1e-3) / 1e9
    e2e_value = world * kv_bytes_per_rank / (e2e_max * 1e-3) / 1e9
    return value, e2e_value, ms_max, e2e_max


# ---------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The float64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    # a step: the five grid shapes at batch 1, seq_len 4096 (bounded sample)
    steps, warm = args.steps, args.warmup
    per_step = []
    total_bytes = 0
    desc = ""
    for i in range(warm + steps):
        b, s, desc = oracle_sample(1e9, lens=[4096],
                                   device="cuda" if torch.cuda.is_available() else "cpu")
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
def kernels_per_call(pa, c):
    """Kernels one decode call of the cell launches, as the library reports it for the
    cell's tensors on this device: the decode grid, plus the merge grid unless the
    context fits one split or its splits merge inside their thread-block clusters."""
    x = c.insts[0]
    return pa.kernel_count(x.q, x.k, x.v, x.bt, x.sl, c.scale, max_seq_len=c.max_len,
                           window=c.window, total_tokens=c.total_tokens)


def steady_state_us(pa, cell, stream, reps_target_ms=3.0):
    """us/call of back-to-back calls rotating over cache copies (graph replay)."""
    n = len(cell.insts)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(n):
            cell.call(pa, stream, i)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                cell.call(pa, stream, i)
        g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        stream.synchronize()
        one = e0.elapsed_time(e1)
        reps = max(3, int(math.ceil(reps_target_ms / max(one, 1e-3))))
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / (reps * n)
    del g
    return 1e3 * ms


def attach_workspaces(pa, lib, cells, dev):
    """One zeroed workspace per cell, so that a captured graph has fixed addresses."""
    import ctypes
    for c in cells:
        x = c.insts[0]
        a = pa.make_args(x.q, x.k, x.v, x.bt, x.sl, x.out, c.scale, c.max_len, 0, c.window,
                         FP8_SCALE, FP8_SCALE, total_tokens=c.total_tokens)
        nbytes = lib.pa_decode_ex_workspace_bytes(ctypes.byref(a))
        c.ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)


def measure_curve(pa, cells, stream, peak):
    """Steady-state µs/call of every cell (or group: the hybrid's 16 layers of one
    context length form one decode step), outside the timed region."""
    curve = []
    groups = {}
    for c in cells:  # the hybrid's 16 layers of one length form one group
        key = c.tag.split(" layer=")[0]
        groups.setdefault(key, []).append(c)
    for key, members in groups.items():
        c = members[0]
        c.add_copies(max(1, min(256, -(-ROTATE_BYTES // max(1, c.kv_bytes())))))
        us = steady_state_us(pa, c, stream)
        gbs = c.kv_bytes() / (us * 1e-6) / 1e9
        S, P = pa.plan(c.B, c.Hq, c.Hkv, c.D, c.bs, c.max_len, window=c.window, kv_fp8=c.fp8,
                       total_tokens=c.total_tokens)
        entry = {"cell": key, "us_per_call": round(us, 3), "kv_gbs": round(gbs, 1),
                 "frac": round(gbs / peak, 4), "splits": S, "copies": len(c.insts)}
        if len(members) == 16:
            # the hybrid's 16 full-attention layers are one decode step; its calls are
            # independent, so the step is 16 back-to-back calls over distinct caches
            entry["ms_per_step_16_layers"] = round(16 * us / 1000.0, 4)
        curve.append(entry)
        del c.insts[1:]
        torch.cuda.empty_cache()
    return curve


def curve_summary(curve):
    """The batch-1 and mixed-batch cells of the curve by context length."""
    out = {}
    for c in curve:
        m = re.match(r"hybrid L=(\d+)$", c["cell"])
        if m:
            out.setdefault("hybrid_us_per_call", {})[m.group(1)] = c["us_per_call"]
            out.setdefault("hybrid_frac", {})[m.group(1)] = c["frac"]
            out.setdefault("hybrid_ms_per_step_16_layers", {})[m.group(1)] = \
                c.get("ms_per_step_16_layers")
        m = re.match(r"(\d+/\d+) B=1 L=(\d+)$", c["cell"])
        if m:
            out.setdefault(f"batch1_{m.group(1)}_frac", {})[m.group(2)] = c["frac"]
        if c["cell"].startswith("mixed"):
            out["mixed_frac"] = c["frac"]
            out["mixed_us_per_call"] = c["us_per_call"]
        m = re.match(r"fp8 hybrid L=(\d+)$", c["cell"])
        if m:
            out.setdefault("fp8_hybrid_us_per_call", {})[m.group(1)] = c["us_per_call"]
            out.setdefault("fp8_hybrid_frac", {})[m.group(1)] = c["frac"]
    for L, us in out.get("fp8_hybrid_us_per_call", {}).items():
        bf = out.get("hybrid_us_per_call", {}).get(L)
        if bf:
            out.setdefault("fp8_over_bf16_hybrid_time", {})[L] = round(us / bf, 3)
    return out


def time_step(pa, cells, stream, steps, warmup):
    """ms per step of all cells' calls captured as one CUDA graph (CUDA events on the
    launching stream, `steps` replays after `warmup`)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in cells:
            c.call(pa, stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in cells:
                c.call(pa, stream)
        for _ in range(warmup):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    del g
    return e0.elapsed_time(e1) / steps


def run_ours(args, rank, world, local_rank):
    import ctypes
    import paged_kv_attention_pa_gb300 as pa
    from paged_kv_attention_pa_gb300 import build as pa_build
    pa_build.build()
    lib = pa.load()

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cells, desc = build_workload(args.workload, dev, seed=args.seed + 1000 * rank,
                                 cell_spec=args.cell)
    stream = torch.cuda.Stream(dev)
    attach_workspaces(pa, lib, cells, dev)
    torch.cuda.synchronize()

    def step_eager():
        for c in cells:
            c.call(pa, stream)

    # warm-up (also loads modules and sets the shared-memory opt-in)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_eager()
    stream.synchronize()
    for c in cells:
        assert torch.isfinite(c.insts[0].out).all(), f"non-finite output in {c.tag}"
        assert pa.read_device_errors(c.ws, stream) == 0, f"device error in {c.tag}"

    # the step as one CUDA graph
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step_eager()
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()

    # ---------------- timed region: K graph replays
    clocks = None
    if rank == 0:
        clocks = NvmlSampler(dev)
        if not clocks.start():
            clocks = ClockSampler(dev.index)
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
    clk = clocks.stop() if clocks else None
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = starts[0].elapsed_time(ends[-1])
    del graph

    # ---------------- end to end through the public API with host buffers
    # Every step copies all cells' q, block tables and seq_lens from one pinned host
    # buffer into one device buffer (the calls take views of it), runs every call
    # through pa.decode, and copies all outputs back in one transfer. The KV caches
    # stay resident: they are the model's state, not a per-step input.
    def carve(tensors):  # 256-byte aligned offsets of the tensors in one buffer
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += -(-(t.numel() * t.element_size()) // 256) * 256
        return offs, max(n, 256)

    def view(buf, off, like):
        nb = like.numel() * like.element_size()
        return buf[off:off + nb].view(like.dtype).view(like.shape)

    ins = [t for c in cells for t in (c.insts[0].q, c.insts[0].bt, c.insts[0].sl)]
    outs = [c.insts[0].out for c in cells]
    in_offs, in_bytes = carve(ins)
    out_offs, out_bytes = carve(outs)
    h_in = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    h_out = torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True)
    d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    for t, o in zip(ins, in_offs):
        view(h_in, o, t).copy_(t)
    e2e_args = [tuple(view(d_in, in_offs[3 * i + j], ins[3 * i + j]) for j in range(3)) +
                (view(d_out, out_offs[i], outs[i]),) for i in range(len(cells))]
    h2d, d2h = in_bytes, out_bytes

    def step_e2e():
        d_in.copy_(h_in, non_blocking=True)
        for c, (q, bt, sl, o) in zip(cells, e2e_args):
            c.call_with(pa, stream, q, bt, sl, o)
        h_out.copy_(d_out, non_blocking=True)

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
    value, e2e_value, ms_step_max, e2e_max = aggregate_over_ranks(kv, ms_step, e2e_ms, world, dev)
    if rank != 0:
        return

    # ---------------- steady-state curve (outside the timed region)
    peak, peak_kind = load_peaks()
    curve = []
    fp8_grid = None
    if not args.no_curve:
        curve = measure_curve(pa, cells, stream, peak)
        if args.workload == "grid":
            # Beside the grid: the hybrid full-attention layer (batch 1, 4 KV heads, head
            # 256, block 784) at every context length as 16-layer steps, and the mixed
            # serving batch, each in steady state like the grid's cells.
            extra = build_workload("hybrid", dev, seed=args.seed + 5000)[0] + \
                build_workload("mixed", dev, seed=args.seed)[0]
            attach_workspaces(pa, lib, extra, dev)
            curve += measure_curve(pa, extra, stream, peak)
            del extra
            torch.cuda.empty_cache()
            # FP8 E4M3 caches: the hybrid layer at 4K / 16K / 32K (steady state, as
            # above) and the grid step (one graph of the 60 calls, like the headline)
            extra = build_workload("hybrid", dev, seed=args.seed + 7000, fp8=True,
                                   lens=[4096, 16384, 32768])[0]
            attach_workspaces(pa, lib, extra, dev)
            curve += measure_curve(pa, extra, stream, peak)
            del extra
            grid8 = build_workload("grid", dev, seed=args.seed + 9000, fp8=True)[0]
            attach_workspaces(pa, lib, grid8, dev)
            ms8 = time_step(pa, grid8, stream, max(args.steps, 10), args.warmup)
            kv8 = sum(c.kv_bytes() for c in grid8)
            fp8_grid = {"ms_per_step": round(ms8, 4), "kv_gbs": round(kv8 / (ms8 * 1e-3) / 1e9, 1),
                        "frac": round(kv8 / (ms8 * 1e-3) / 1e9 / peak, 4),
                        "kv_bytes_per_step": kv8}
            del grid8
            torch.cuda.empty_cache()

    linearity = hybrid_linearity(curve)

    budget = float(os.environ.get("PA_BENCH_CPU_BUDGET_S", "12"))
    cb_bytes, cb_s, cb_desc = oracle_sample(budget, device=dev)
    achieved = alg / (ms_step_max * 1e-3) / 1e9
    Ds = {c.D for c in cells}
    traffic, traffic_note = (traffic_per_call(alg / len(cells), Ds.pop(),
                                              "fp8" if KV_FP8 else "bf16")
                             if len(Ds) == 1 else (None, "cells of several head_dims"))
    line = {
        "impl": "ours", "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 q/out, fp8-e4m3 KV" if KV_FP8 else "bf16",
        "data": "synthetic",
        "config": dict(desc, **{
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "kv_dtype": "fp8_e4m3" if KV_FP8 else "bf16",
            "l2": "inputs larger than L2: each step reads every cell's own cache once "
                  f"({kv / 2**30:.2f} GiB of distinct KV per step)",
            "timed": "CUDA graph of the whole step, replayed K times, CUDA events",
            "kv_bytes_per_step": kv}),
        "gpu_launches": sum(kernels_per_call(pa, c) for c in cells) * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_source": traffic_note,
                     "peak_kind": peak_kind,
                     "kernel": "pa::decode_kernel (+ pa::merge_kernel where the splits do not merge in their clusters)",
                     "alg_bytes_per_launch": round(alg / len(cells)),
                     "avg_launch_us": round(1e3 * ms_step_max / len(cells), 3),
                     "launch_timing": "timed region / decode calls (graph replay, "
                                      "programmatic dependent launch between calls)"},
        "cpu_baseline": {"value": round(cb_bytes / cb_s / 1e9, 4), "unit": "GB/s",
                         "cores": cpu_threads(), "kind": "oracle", "sample": cb_desc},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "what": "per step: one pinned H2D of every cell's q, block table and "
                        "seq_lens; eager pa.decode per cell (Python binding, C ABI); one D2H "
                        "of every output (KV caches resident)"},
        "clocks": clk,
        "step_ms_min_med_max": [round(min(step_ms), 4), round(statistics.median(step_ms), 4),
                                round(max(step_ms), 4)],
        "curve": curve,
    }
    if linearity:
        line["linearity"] = linearity
    if curve:
        line["summary"] = curve_summary(curve)
        if fp8_grid:
            line["summary"]["fp8_grid_step"] = fp8_grid
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="grid",
                    choices=["grid", "hybrid", "mixed", "first", "cell", "window", "rows"])
    ap.add_argument("--cell", default=None, help="Hq,Hkv,B,L,D,block_size for --workload cell")
    ap.add_argument("--no-curve", action="store_true", help="skip the steady-state curve")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="cache element type (fp8 = E4M3 with a per-tensor scale)")
    args = ap.parse_args()
    global KV_FP8
    KV_FP8 = args.kv_dtype == "fp8"
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
