"""Benchmark of the gated W4 + low-rank compensated linear on GB300.

One step = one pass of the decode hot path over the Llama-7B decode workload:
the three decoder linear shapes (K x N = 4096x4096, 4096x11008, 11008x4096),
int4 group-128 asymmetric weights with uint4 zero points, rank-32
compensator, each at M = 1, 4, 16 and 64 tokens (x ~ N(0,1) with 1% outlier
channels x20): 12 fused decode launches.  The headline value is algorithmic
HBM bytes of those 12 calls per second (GB/s).  A second measurement covers
the prefill path (TFLOP/s) on the prefill workload (same shapes, M = 512,
2048, 8192).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own replica of the workload (weak scaling);
rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode fused W4+comp GB/s (% HBM peak); prefill TFLOP/s (% bf16 peak)"
DECODE_SHAPES = [(4096, 4096), (4096, 11008), (11008, 4096)]      # (K, N)
DECODE_M = [1, 4, 16, 64]
PREFILL_M = [512, 2048, 8192]
G, SYM, RANK, OUTLIERS = 128, False, 32, 0.01
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the library serves decode calls of M >= 17 tokens with its tensor-core kernel
# (decode_tc.cu), smaller ones with the warp-level kernel (decode.cu)
TC_MIN_M = 17
N_CHECK = 4096            # leading outputs compared between the host copy and the device after the e2e loop
DRAM_SUMMARY = os.path.join(ROOT, "profiles", "decode_dram_bytes.json")


def decode_kernel_name(M: int) -> str:
    return "decode_tc_kernel" if M >= TC_MIN_M else "decode_kernel"


# the files each decode kernel is compiled from (its own and the shared headers)
KERNEL_SOURCES = {"decode_kernel": ("decode.cu", "common.cuh"),
                  "decode_tc_kernel": ("decode_tc.cu", "common.cuh", "sm100_ptx.cuh", "tmap.h")}


def code_digest(text: str) -> str:
    """Digest of C++/CUDA source with comments and whitespace removed, so an
    edit to the comments alone does not mark the counters stale."""
    import hashlib
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def source_digest(name: str) -> str:
    with open(os.path.join(ROOT, "quantized_gemm_error_gb300", "csrc", name)) as f:
        return code_digest(f.read())


def measured_traffic(kernel: str, cases):
    """DRAM bytes per launch of `kernel` over the bench's cases, from the
    committed ncu summary -- only while the kernel source is the one the
    counters were taken with (else None)."""
    if not os.path.exists(DRAM_SUMMARY):
        return None
    d = json.load(open(DRAM_SUMMARY))
    for src in KERNEL_SOURCES[kernel]:
        if d.get("sources", {}).get(src) != source_digest(src):
            return None
    per = [d["launches"].get(f"{kernel} K={c['K']} N={c['N']} M={c['M']}") for c in cases]
    if not per or any(v is None for v in per):
        return None
    return round(float(np.mean(per)))


def decode_bytes(K: int, N: int, M: int, r: int = RANK, comp: bool = True) -> int:
    """Algorithmic HBM bytes of one decode call: codes, scales, zero points,
    compensator factors (A, w_g, B), tokens in, outputs out."""
    ng = K // G
    b = N * K // 2 + N * ng * 2 + N * ((ng + 1) // 2) + M * K * 2 + M * N * 2
    if comp:
        b += (r + 1) * K * 2 + N * r * 2
    return b


def prefill_flops(K: int, N: int, M: int, r: int = RANK, comp: bool = True) -> int:
    f = 2 * M * N * K
    if comp:
        f += 2 * M * r * (K + N) + 2 * M * K
    return f


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
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

    def summary(self):
        mhz, maxmhz, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                maxmhz.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(mhz)), "sm_max_mhz": float(max(maxmhz)),
                "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- oracle

def oracle_case(K, N, M, seed, rows=None):
    import oracle
    from quantized_gemm_error_gb300.inputs import make_layer, make_tokens
    lay, rng = make_layer(N, K, RANK, seed=seed)
    x = make_tokens(rng, M, K, outlier_frac=OUTLIERS)
    q, s, z = oracle.quantize_pack(lay.W, G, SYM)
    L = dict(N=N, K=K, G=G, sym=SYM, qweight=q, scales=s, zeros=z, r=RANK, A=lay.A, B=lay.B, w_g=lay.w_g,
             b_g=0.0, alpha=1.0, comp_enabled=1)
    return L, x


def time_oracle(cases, nthreads):
    """Runs the oracle (as it stands) on each (layer, x, rows) case; returns
    (seconds, algorithmic bytes covered)."""
    import oracle
    t0 = time.perf_counter()
    nbytes = 0.0
    for L, x, rows in cases:
        oracle.linear(L, x, n_idx=rows, nthreads=nthreads)
        K, N, M = L["K"], L["N"], x.shape[0]
        frac = 1.0 if rows is None else len(rows) / N
        nbytes += decode_bytes(K, N, M) * frac
    return time.perf_counter() - t0, nbytes


def host_threads() -> int:
    """Threads for the oracle: the CPUs this process may run on (its affinity
    set), not every CPU of the machine."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(row_fraction: float = 1.0):
    """The oracle timed on this host's cores on a bounded sample of the decode
    step: every (shape, M) call of the step, a fixed seeded subset of output
    rows (row_fraction of N), fp64 accumulation; throughput scaled to the
    metric's unit (algorithmic bytes of the rows covered per second)."""
    nthreads = host_threads()
    cases = []
    rng = np.random.default_rng(0)
    for (K, N) in DECODE_SHAPES:
        for M in DECODE_M:
            L, x = oracle_case(K, N, M, seed=K + N)
            rows = np.sort(rng.choice(N, size=max(16, int(N * row_fraction)), replace=False)).astype(np.int32)
            cases.append((L, x, rows))
    secs, nbytes = time_oracle(cases, nthreads)
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": nthreads, "host_cpus": os.cpu_count(),
            "kind": "oracle",
            "sample": f"the 12 decode calls of one step, {row_fraction:.4g} of each layer's output rows "
                      f"(seeded), fp64 accumulation, {secs:.1f} s"}


def decode_workload_config() -> dict:
    """The decode workload's keys both arms report: the layers, token counts,
    quantisation format, rank and the algorithmic bytes of one step."""
    return {"workload": "llama7b_decode_g128_r32", "shapes_KxN": [list(s) for s in DECODE_SHAPES],
            "M": DECODE_M, "group_size": G, "symmetric": SYM, "rank": RANK,
            "calls_per_step": len(DECODE_SHAPES) * len(DECODE_M),
            "bytes_per_step": sum(decode_bytes(K, N, M) for (K, N) in DECODE_SHAPES for M in DECODE_M)}


# ------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    nthreads = host_threads()
    # size each step's sample so the whole run stays within --ref-budget-s
    # (two minutes by default)
    probe_L, probe_x = oracle_case(4096, 4096, 1, seed=1)
    rows = np.arange(64, dtype=np.int32)
    dt, _ = time_oracle([(probe_L, probe_x, rows)], nthreads)
    per_row_m1 = dt / 64
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    cases = []
    for (K, N) in DECODE_SHAPES:
        for M in DECODE_M:
            L, x = oracle_case(K, N, M, seed=K + N)
            cases.append((L, x))
    # cost of one row of one call ~ per_row_m1 * (K/4096) * (1 + M)/2; pick rows per case
    est = sum(per_row_m1 * (L["K"] / 4096) * (1 + x.shape[0]) / 2 for L, x in cases)
    rows_per_case = int(max(1, min(512, budget / max(est, 1e-9))))
    rng = np.random.default_rng(0)
    step_cases = [(L, x, np.sort(rng.choice(L["N"], rows_per_case, replace=False)).astype(np.int32))
                  for L, x in cases]
    # every call also forms its tokens' rank-r code over all of K, whatever
    # rows it covers: when even one row per call does not fit a step's share
    # of the time, a step takes a rotating block of the 12 calls instead
    per_call = len(step_cases)
    if rows_per_case == 1:
        t_full, _ = time_oracle(step_cases, nthreads)
        if t_full > budget:
            per_call = max(1, int(len(step_cases) * budget / t_full))
    blocks = [[step_cases[(i + j) % len(step_cases)] for j in range(per_call)]
              for i in range(0, len(step_cases), per_call)]
    for i in range(args.warmup):
        time_oracle(blocks[i % len(blocks)], nthreads)
    total_s, total_b = 0.0, 0.0
    for i in range(args.steps):
        s, b = time_oracle(blocks[i % len(blocks)], nthreads)
        total_s += s
        total_b += b
    value = total_b / total_s / 1e9
    if per_call == len(step_cases):
        sample = (f"each step: the 12 decode calls of the step on {rows_per_case} seeded output rows per "
                  f"call, fp64 accumulation")
    else:
        sample = (f"each step: {per_call} of the step's 12 decode calls in rotation, {rows_per_case} seeded "
                  f"output row per call, fp64 accumulation")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(decode_workload_config(), parallelism="rank 0 on the host cores"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "host_cpus": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# -------------------------------------------------------------------- ours

def build_decode(torch, spear, device, l2_bytes):
    """The decode workload's three layers, each in `ncopy` distinct copies on
    the device.  ncopy is the smallest multiple of the 4 token counts whose
    copies of the smallest layer add up to at least 4x L2: every call of a
    step then reads a weight copy that at least 4x L2 of other weights of the
    same shape have passed through since its last use, so its weights come
    from HBM."""
    from quantized_gemm_error_gb300.inputs import make_layer, make_tokens

    def dev16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    base = []
    for (K, N) in DECODE_SHAPES:
        lay, rng = make_layer(N, K, RANK, seed=K + N)
        q, s, z = spear.spear_pack_w4(torch.from_numpy(lay.W).to(device), G, SYM)
        L = spear.W4Layer(N, K, G, SYM, q, s, z, RANK, dev16(lay.A), dev16(lay.B), dev16(lay.w_g), 0.0, 1.0, True)
        xs = {M: make_tokens(rng, M, K, outlier_frac=OUTLIERS) for M in DECODE_M}
        base.append((K, N, L, xs))
    min_bytes = min(decode_bytes(K, N, 0) for K, N, _, _ in base)
    nm = len(DECODE_M)
    ncopy = int(nm * np.ceil(np.ceil(4.0 * l2_bytes / min_bytes) / nm))
    copies = [base]
    for _ in range(ncopy - 1):
        cp = []
        for K, N, L, xs in base:
            L2 = spear.W4Layer(N, K, G, SYM, L.qweight.clone(), L.scales.clone(), L.zeros.clone(), RANK,
                               L.A.clone(), L.B.clone(), L.w_g.clone(), 0.0, 1.0, True)
            cp.append((K, N, L2, xs))
        copies.append(cp)
    set_bytes = sum(decode_bytes(K, N, 0) for K, N, _, _ in base)
    return copies, ncopy, set_bytes


def step_copy(t: int, m_index: int, ncopy: int) -> int:
    """Weight copy read by the call with token-count index m_index in step t:
    the 4 calls of one shape in a step read 4 different copies, and each copy
    comes round again after ncopy / 4 steps."""
    return (len(DECODE_M) * t + m_index) % ncopy


def run_ours(args, world, rank, local):
    import torch

    from quantized_gemm_error_gb300 import spear
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks, peak_kind = load_peaks()
    props = torch.cuda.get_device_properties(device)
    l2_bytes = getattr(props, "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20

    copies, ncopy, set_bytes = build_decode(torch, spear, device, l2_bytes)
    # consecutive decode calls never write each other's weights: let each
    # launch overlap the tail of the one before it
    spear.spear_set_launch_overlap(True)
    stream = torch.cuda.Stream(device)
    xs_dev = {}
    ys = {}
    calls = []   # (K, N, M) per call in a step
    for K, N, L, xs in copies[0]:
        for M in DECODE_M:
            xs_dev[(K, M)] = torch.from_numpy(xs[M].view(np.int16)).view(torch.bfloat16).to(device)
            ys[(N, M)] = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            calls.append((K, N, M))
    ws_bytes = max(spear.spear_decode_workspace_bytes(L, M) for _, _, L, _ in copies[0] for M in DECODE_M)
    ws = spear.new_workspace(ws_bytes, device)
    torch.cuda.synchronize()              # inputs made on the default stream; calls run on `stream`
    step_bytes = sum(decode_bytes(K, N, M) for K, N, M in calls)

    def layer_of(cp, K, N):
        return [l for (k, n, l, _) in copies[cp] if (k, n) == (K, N)][0]

    nphase = ncopy // len(DECODE_M)          # steps until the copy pattern repeats

    def step(t, comp=True):
        for K, N, _, _ in copies[0]:
            for mi, M in enumerate(DECODE_M):
                L = layer_of(step_copy(t, mi, ncopy), K, N)
                Lc = L if comp else L.with_comp(False)
                spear.spear_linear_decode(Lc, xs_dev[(K, M)], y=ys[(N, M)], workspace=ws, stream=stream)

    # warm the library's launch plans, then capture one graph per step phase
    with torch.cuda.stream(stream):
        for t in range(nphase):
            step(t)
            step(t, comp=False)
    torch.cuda.synchronize()
    assert spear.spear_get_device_status() == 0
    graphs, launch_mode = [], "cuda-graph"
    try:
        for t in range(nphase):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(t)
            graphs.append(g)
    except Exception as e:  # pragma: no cover - capture unsupported
        graphs, launch_mode = [], f"eager ({type(e).__name__})"
        torch.cuda.synchronize()

    def replay(i):
        if graphs:
            graphs[i % nphase].replay()
        else:
            with torch.cuda.stream(stream):
                step(i % nphase)

    for i in range(max(3, args.warmup)):
        replay(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(world)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                replay(i)
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    t_ms = e0.elapsed_time(e1)
    t_max = reduce_max(t_ms, world)
    assert spear.spear_get_device_status(stream) == 0
    value = world * args.steps * step_bytes / (t_max / 1e3) / 1e9

    # per-call breakdown: for each call of the step, one graph holding that
    # call on every weight copy (consecutive launches overlap as in the step);
    # comp on vs off
    # the pages' vector gate (hidden width 8 on the rank-32 code) on the same
    # weights, against the task's scalar gate and the plain layer
    import dataclasses
    gen = torch.Generator(device=device)
    gen.manual_seed(0)
    vg = dict(gate_w1=torch.randn(8, RANK, generator=gen, device=device) * (3.0 / RANK ** 0.5),
              gate_c1=torch.randn(8, generator=gen, device=device) * 0.1,
              gate_w2=torch.randn(RANK, 8, generator=gen, device=device) / 8 ** 0.5,
              gate_c2=torch.randn(RANK, generator=gen, device=device))
    cases = []
    for (K, N, M) in calls:
        res = {}
        for comp in (True, False, "vector"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for cp in range(ncopy):
                    L = layer_of(cp, K, N)
                    Lc = (L if comp is True else L.with_comp(False) if comp is False
                          else dataclasses.replace(L, w_g=None, **vg))
                    spear.spear_linear_decode(Lc, xs_dev[(K, M)], y=ys[(N, M)], workspace=ws, stream=stream)
            reps = 5
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            with torch.cuda.stream(stream):
                for i in range(reps):
                    g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            res[comp] = a.elapsed_time(b) / (reps * ncopy) * 1e3
        gbs = decode_bytes(K, N, M) / res[True] / 1e3
        cases.append({"K": K, "N": N, "M": M, "kernel": decode_kernel_name(M), "us": round(res[True], 3),
                      "GB_s": round(gbs, 1),
                      "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 4),
                      "frac_hbm_8000": round(gbs / 8000.0, 4),
                      "plain_us": round(res[False], 3), "comp_overhead": round(res[True] / res[False] - 1, 4),
                      "vector_gate_us": round(res["vector"], 3),
                      "vector_gate_overhead": round(res["vector"] / res[False] - 1, 4)})
    tot_on = sum(c["us"] for c in cases)
    tot_off = sum(c["plain_us"] for c in cases)

    # end to end through the public API with host buffers (pinned): per step one
    # host-to-device copy of all the step's tokens (one pinned buffer), the 12
    # decode calls on views of it, and one device-to-host copy of their 12
    # outputs, captured as one CUDA graph per weight copy (as a serving loop
    # would issue it); the copies stay inside the timed region every step
    call_list = [(K, N, M) for (K, N) in DECODE_SHAPES for M in DECODE_M]
    x_off, y_off, xo, yo = {}, {}, 0, 0
    for (K, N, M) in call_list:
        x_off[(K, N, M)] = xo
        y_off[(K, N, M)] = yo
        xo += M * K
        yo += M * N
    # two slots of device buffers (and of host outputs), so that a step's
    # inputs can travel in while the step before it computes and its outputs
    # travel out while the step after it computes, as a serving loop would
    # pipeline them: every step still copies its own inputs from pinned host
    # memory and reads its own outputs back inside the timed region
    h_x = torch.empty(xo, dtype=torch.bfloat16).pin_memory()
    h_y = [torch.empty(yo, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    d_x = [torch.empty(xo, dtype=torch.bfloat16, device=device) for _ in range(2)]
    d_y = [torch.empty(yo, dtype=torch.bfloat16, device=device) for _ in range(2)]
    for (K, N, M) in call_list:
        h_x[x_off[(K, N, M)]:x_off[(K, N, M)] + M * K].copy_(xs_dev[(K, M)].reshape(-1).cpu())
    h2d, d2h = xo * 2, yo * 2
    torch.cuda.synchronize()
    # the 12 calls of a step, one graph per (weight-copy phase, slot)
    e2e_graphs = {}
    for t in range(nphase):
        for sl in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for (K, N, M) in call_list:
                    L = layer_of(step_copy(t, DECODE_M.index(M), ncopy), K, N)
                    xv = d_x[sl][x_off[(K, N, M)]:x_off[(K, N, M)] + M * K].view(M, K)
                    yv = d_y[sl][y_off[(K, N, M)]:y_off[(K, N, M)] + M * N].view(M, N)
                    spear.spear_linear_decode(L, xv, y=yv, workspace=ws, stream=stream)
            e2e_graphs[(t, sl)] = g
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event()
    computed = [ev(), ev()]                # slot's last compute done
    arrived = [ev(), ev()]                 # slot's inputs in place
    returned = [ev(), ev()]                # slot's outputs read back

    def e2e_run(nsteps):
        for sl in range(2):                # every slot free
            computed[sl].record(stream)
            returned[sl].record(s_out)
        for i in range(nsteps):
            sl = i % 2
            s_in.wait_event(computed[sl])                  # the step two back is done with this slot
            with torch.cuda.stream(s_in):
                d_x[sl].copy_(h_x, non_blocking=True)
            arrived[sl].record(s_in)
            stream.wait_event(arrived[sl])
            stream.wait_event(returned[sl])                # its outputs two steps back are read
            with torch.cuda.stream(stream):
                e2e_graphs[(i % nphase, sl)].replay()
            computed[sl].record(stream)
            s_out.wait_event(computed[sl])
            with torch.cuda.stream(s_out):
                h_y[sl].copy_(d_y[sl], non_blocking=True)
            returned[sl].record(s_out)
        stream.wait_event(returned[(nsteps - 1) % 2])
        stream.wait_event(returned[nsteps % 2])

    e2e_steps = max(3, min(args.steps, 2000))
    e2e_run(2 * nphase)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_run(e2e_steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b), world)
    e2e_value = world * e2e_steps * step_bytes / (e2e_ms / 1e3) / 1e9
    last = (e2e_steps - 1) % 2
    assert torch.equal(h_y[last][:N_CHECK].to(torch.float32), d_y[last][:N_CHECK].cpu().to(torch.float32))
    # the same steps with each step's copies and calls in series on one
    # stream (no overlap between steps), reported beside it
    torch.cuda.synchronize()
    barrier(world)
    a.record(stream)
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            d_x[0].copy_(h_x, non_blocking=True)
            e2e_graphs[(i % nphase, 0)].replay()
            h_y[0].copy_(d_y[0], non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_serial_value = world * e2e_steps * step_bytes / (reduce_max(a.elapsed_time(b), world) / 1e3) / 1e9
    last = 0
    assert torch.equal(h_y[last][:N_CHECK].to(torch.float32), d_y[last][:N_CHECK].cpu().to(torch.float32))

    prefill = None
    if not args.no_prefill:
        try:
            prefill = run_prefill(torch, spear, device, stream, peaks)
        except Exception as e:  # the decode line still prints; the failure is reported in it
            prefill = {"error": f"{type(e).__name__}: {e}"}
    # the other two workloads, on rank 0 (a few seconds of GPU time each)
    stack = llama70b = None
    del copies, graphs, e2e_graphs
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_extra:
        try:
            stack = stack_section(torch, spear, device, peaks, steps=10, warmup=3)
        except Exception as e:
            stack = {"error": f"{type(e).__name__}: {e}"}
        try:
            llama70b = llama70b_section(torch, spear, device, stream, peaks, l2_bytes)
        except Exception as e:
            llama70b = {"error": f"{type(e).__name__}: {e}"}

    # roofline of the kernel with the largest share of the step: algorithmic
    # bytes per launch over its mean launch time (CUDA events, graph replays)
    by_kernel = {}
    for c in cases:
        by_kernel.setdefault(c["kernel"], []).append(c)
    dominant = max(by_kernel, key=lambda k: sum(c["us"] for c in by_kernel[k]))
    dcases = by_kernel[dominant]
    d_bytes = sum(decode_bytes(c["K"], c["N"], c["M"]) for c in dcases) / len(dcases)
    d_us = sum(c["us"] for c in dcases) / len(dcases)
    ach = d_bytes / d_us / 1e3
    shares = {k: round(sum(c["us"] for c in v) / tot_on, 4) for k, v in by_kernel.items()}

    result = None
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baseline()
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {**decode_workload_config(),
                       "l2": f"every call of a step reads its own weight copy; each layer rotates through "
                             f"{ncopy} copies ({ncopy * set_bytes / 1e6:.0f} MB of weights in all; the smallest "
                             f"layer's copies alone >= 4x L2 {l2_bytes / 1e6:.0f} MB), per-call timings likewise",
                       "weight_copies": ncopy,
                       "launch": launch_mode, "launch_overlap": True, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "peak_kind": peak_kind,
                         "frac_of_8000": round(ach / 8000.0, 4),
                         "traffic": measured_traffic(dominant, dcases),
                         "algorithmic_bytes_per_launch": round(d_bytes), "launch_us": round(d_us, 3),
                         "time_share": shares},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "copies": "every step's H2D and D2H inside the timed region, on two copy streams, "
                              "overlapping the neighbouring steps' kernels (two buffer slots)",
                    "serial_value": round(e2e_serial_value, 2)},
            "gpu_launches": args.steps * len(calls),
            "clocks": clk.summary(),
            "comp_overhead_step": round(tot_on / tot_off - 1, 4),
            "vector_gate_overhead_step": round(sum(c["vector_gate_us"] for c in cases) / tot_off - 1, 4),
            "decode_cases": cases,
            "prefill": prefill,
            "stack": stack,
            "llama70b": llama70b,
        }
        print(json.dumps(result), flush=True)
    return result


def run_prefill(torch, spear, device, stream, peaks):
    """Prefill TFLOP/s on the prefill workload (3 shapes x M in 512/2048/8192),
    fused and concurrent-stream modes and the plain W4 GEMM."""
    from quantized_gemm_error_gb300.inputs import make_layer, make_tokens

    def dev16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    aux = torch.cuda.Stream(device)
    out = []
    tot_flops = 0.0
    tot_s = 0.0
    for (K, N) in DECODE_SHAPES:
        lay, rng = make_layer(N, K, RANK, seed=K + N + 1)
        q, s, z = spear.spear_pack_w4(torch.from_numpy(lay.W).to(device), G, SYM)
        L = spear.W4Layer(N, K, G, SYM, q, s, z, RANK, dev16(lay.A), dev16(lay.B), dev16(lay.w_g), 0.0, 1.0, True)
        for M in PREFILL_M:
            x = dev16(make_tokens(rng, M, K, outlier_frac=OUTLIERS))
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = spear.new_workspace(max(spear.spear_prefill_workspace_bytes(L, M, m)
                                         for m in (spear.PREFILL_FUSED, spear.PREFILL_STREAM)), device, zero=False)
            torch.cuda.synchronize()          # inputs made on the default stream; calls run on `stream`
            res = {}
            for name, Lc, mode in (("fused", L, spear.PREFILL_FUSED), ("stream", L, spear.PREFILL_STREAM),
                                   ("plain", L.with_comp(False), spear.PREFILL_FUSED)):
                def call():
                    spear.spear_linear_prefill(Lc, x, y=y, mode=mode, workspace=ws, stream=stream, stream_aux=aux)
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        call()
                torch.cuda.synchronize()
                reps = max(3, int(2e13 / prefill_flops(K, N, M)))
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    for _ in range(reps):
                        call()
                    b.record(stream)
                torch.cuda.synchronize()
                res[name] = a.elapsed_time(b) / reps * 1e3
            assert spear.spear_get_device_status(stream) == 0
            best = min(res["fused"], res["stream"])
            fl = prefill_flops(K, N, M)
            tflops = fl / best / 1e6
            tot_flops += fl
            tot_s += best * 1e-6
            out.append({"K": K, "N": N, "M": M, "fused_us": round(res["fused"], 1), "stream_us": round(res["stream"], 1),
                        "plain_us": round(res["plain"], 1), "TFLOP_s": round(tflops, 1),
                        "frac_bf16_burst": round(tflops / peaks["bf16_tflops"], 4),
                        "comp_overhead": round(best / res["plain"] - 1, 4),
                        "best_mode": "fused" if res["fused"] <= res["stream"] else "stream"})
            del x, y, ws
    agg = tot_flops / tot_s / 1e12
    return {"metric": "prefill TFLOP/s", "value": round(agg, 1), "unit": "TFLOP/s",
            "workload": "llama7b_prefill_g128_r32",
            "roofline": {"bound": "tensor", "achieved": round(agg, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(agg / peaks["bf16_tflops"], 4),
                         "peak_sustained": peaks.get("bf16_tflops_sustained")},
            "cases": out}


def profile_prefill_case(spec: str):
    """One prefill call, repeated, for a profiler to capture (no timing, no JSON):
    --profile-prefill K,N,M,mode,iters with mode 0 auto, 1 fused, 2 stream, 3 plain."""
    import torch
    from quantized_gemm_error_gb300 import spear
    from quantized_gemm_error_gb300.inputs import make_layer, make_tokens
    K, N, M, mode, iters = (int(v) for v in spec.split(","))
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    spear.load()

    def dev16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    lay, rng = make_layer(N, K, RANK, seed=K + N + 1)
    q, s, z = spear.spear_pack_w4(torch.from_numpy(lay.W).to(device), G, SYM)
    L = spear.W4Layer(N, K, G, SYM, q, s, z, RANK, dev16(lay.A), dev16(lay.B), dev16(lay.w_g), 0.0, 1.0, mode != 3)
    x = dev16(make_tokens(rng, M, K, outlier_frac=OUTLIERS))
    torch.cuda.synchronize()
    for _ in range(iters):
        spear.spear_linear_prefill(L, x, mode=spear.PREFILL_FUSED if mode == 3 else mode)
    torch.cuda.synchronize()
    print(f"prefill K={K} N={N} M={M} mode={mode} x{iters}: status {spear.spear_get_device_status()}")


def stack_section(torch, spear, device, peaks, steps: int, warmup: int) -> dict:
    """The Llama-7B 32-block decoder stack (per-channel symmetric int4; rank-64
    compensators on the 4 blocks the selection rule picks): one mixed step of
    chunked prefill (a 1024-token chunk and 32 decode tokens, 1056 tokens
    through all 224 linears on the prefill path) and the 32 decode tokens
    alone on the decode path, each one CUDA graph.  Weights (3.2 GB of int4)
    exceed L2, so every replay streams them from HBM."""
    from quantized_gemm_error_gb300.inputs import workload
    from quantized_gemm_error_gb300.stack import StackStep, build_stack, memory_bytes, select_blocks
    wl = workload("llama7b_stack_sym_r64")
    mask, ranks = select_blocks(wl["blocks"], wl["masked_blocks"], wl["r"], seed=0)
    layers = build_stack(ranks, device, seed=0, recipe="device")
    step = StackStep(layers, wl["prefill_M"][0], wl["decode_M"][0], device, seed=0)
    step.capture()
    out = {}
    for name in ("prefill", "decode"):
        for _ in range(warmup):
            step.replay(name)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(step.stream)
        for _ in range(steps):
            step.replay(name)
        e1.record(step.stream)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / steps            # ms per pass
    status = spear.spear_get_device_status()
    tp, td = out["prefill"] / 1e3, out["decode"] / 1e3
    res = {
        "workload": "llama7b_stack_sym_r64", "blocks": wl["blocks"], "linears": len(layers),
        "compensated_blocks": [int(b) for b in np.flatnonzero(mask)], "rank": wl["r"],
        "prefill_M": step.Mp, "decode_M": step.Md, "launch": "cuda-graph", "steps": steps, "warmup": warmup,
        "l2": "3.2 GB of int4 weights stream from HBM every pass",
        "memory": memory_bytes(ranks),
        "mixed_step": {"ms": round(out["prefill"], 4), "tokens_s": round(step.Mp / tp, 1),
                       "TFLOP_s": round(step.prefill_flops() / tp / 1e12, 1),
                       "frac_bf16_burst": round(step.prefill_flops() / tp / 1e12 / peaks["bf16_tflops"], 4)},
        "decode_step": {"ms": round(out["decode"], 4), "tokens_s": round(step.Md / td, 1),
                        "GB_s": round(step.decode_bytes() / td / 1e9, 1),
                        "frac_hbm": round(step.decode_bytes() / td / 1e9 / peaks["hbm_gbs"], 4)},
        "status": status,
    }
    del step, layers
    torch.cuda.empty_cache()
    return res


def run_stack(args):
    """The decoder stack alone, as its own JSON line (--stack)."""
    import torch
    from quantized_gemm_error_gb300 import spear
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    spear.load()
    spear.spear_set_launch_overlap(True)
    peaks, _ = load_peaks()
    st = stack_section(torch, spear, device, peaks, args.steps, args.warmup)
    tp = st["mixed_step"]["ms"] / 1e3
    line = {
        "metric": "decoder-stack mixed step tokens/s (1056 tokens x 224 linears, prefill path)",
        "value": st["mixed_step"]["tokens_s"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": st["mixed_step"]["ms"], "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {k: st[k] for k in ("workload", "blocks", "linears", "compensated_blocks", "rank", "prefill_M",
                                      "decode_M", "launch", "l2")},
        "memory": st["memory"],
        "prefill_path": {"TFLOP_s": st["mixed_step"]["TFLOP_s"], "frac_bf16_burst": st["mixed_step"]["frac_bf16_burst"]},
        "decode_path": st["decode_step"],
        "gpu_launches": None, "status": st["status"], "seconds_per_step": tp,
    }
    print(json.dumps(line), flush=True)


def llama70b_section(torch, spear, device, stream, peaks, l2_bytes) -> dict:
    """Llama-70B linears (8192x8192, 8192x28672, 28672x8192; int4 group 128
    asymmetric, rank 64, 1 % outlier channels x20): decode GB/s at M in
    {1, 8, 32}, every call on its own weight copy (each shape's copies >= 4x
    L2), and prefill TFLOP/s at M in {256, 512, 1024, 2048, 4096} (fused and
    concurrent-stream modes, the faster one counted), each against the plain
    W4 layer."""
    from quantized_gemm_error_gb300.inputs import make_layer, make_tokens, workload
    wl = workload("llama70b_g128_r64")
    r, Gw, sym, outl = wl["r"], wl["G"], wl["sym"], wl["outlier_frac"]
    assert Gw == G and sym == SYM             # decode_bytes / prefill_flops use the module's format

    def dev16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    aux = torch.cuda.Stream(device)
    dec, pre = [], []
    for (K, N) in wl["shapes"]:
        lay, rng = make_layer(N, K, r, seed=K + N + 7)
        q, s_, z = spear.spear_pack_w4(torch.from_numpy(lay.W).to(device), Gw, sym)
        A, B, wg = dev16(lay.A), dev16(lay.B), dev16(lay.w_g)
        del lay
        L0 = spear.W4Layer(N, K, Gw, sym, q, s_, z, r, A, B, wg, 0.0, 1.0, True)
        wbytes = decode_bytes(K, N, 0, r)
        ncopy = int(np.ceil(4 * l2_bytes / wbytes))
        copies = [L0] + [spear.W4Layer(N, K, Gw, sym, q.clone(), s_.clone(), z.clone(), r, A.clone(), B.clone(),
                                       wg.clone(), 0.0, 1.0, True) for _ in range(ncopy - 1)]
        for M in wl["decode_M"]:
            x = dev16(make_tokens(rng, M, K, outlier_frac=outl))
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = spear.new_workspace(spear.spear_decode_workspace_bytes(L0, M), device)
            torch.cuda.synchronize()
            res = {}
            for comp in (True, False):
                def calls():
                    for L in copies:
                        spear.spear_linear_decode(L if comp else L.with_comp(False), x, y=y, workspace=ws,
                                                  stream=stream)
                with torch.cuda.stream(stream):
                    calls()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    calls()
                g.replay()
                torch.cuda.synchronize()
                reps = 5
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                with torch.cuda.stream(stream):
                    for _ in range(reps):
                        g.replay()
                b.record(stream)
                torch.cuda.synchronize()
                res[comp] = a.elapsed_time(b) / (reps * ncopy) * 1e3
                del g
            assert spear.spear_get_device_status(stream) == 0
            gbs = decode_bytes(K, N, M, r) / res[True] / 1e3
            dec.append({"K": K, "N": N, "M": M, "kernel": decode_kernel_name(M), "us": round(res[True], 3),
                        "GB_s": round(gbs, 1), "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 4),
                        "plain_us": round(res[False], 3), "comp_overhead": round(res[True] / res[False] - 1, 4),
                        "weight_copies": ncopy})
            del x, y, ws
        del copies
        torch.cuda.empty_cache()
        for M in wl["prefill_M"]:
            x = dev16(make_tokens(rng, M, K, outlier_frac=outl))
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = spear.new_workspace(max(spear.spear_prefill_workspace_bytes(L0, M, m)
                                         for m in (spear.PREFILL_FUSED, spear.PREFILL_STREAM)), device, zero=False)
            torch.cuda.synchronize()
            res = {}
            for name, Lc, mode in (("fused", L0, spear.PREFILL_FUSED), ("stream", L0, spear.PREFILL_STREAM),
                                   ("plain", L0.with_comp(False), spear.PREFILL_FUSED)):
                def call():
                    spear.spear_linear_prefill(Lc, x, y=y, mode=mode, workspace=ws, stream=stream, stream_aux=aux)
                with torch.cuda.stream(stream):
                    for _ in range(2):
                        call()
                torch.cuda.synchronize()
                reps = max(2, int(1e13 / prefill_flops(K, N, M, r)))
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    for _ in range(reps):
                        call()
                    b.record(stream)
                torch.cuda.synchronize()
                res[name] = a.elapsed_time(b) / reps * 1e3
            assert spear.spear_get_device_status(stream) == 0
            best = min(res["fused"], res["stream"])
            tfl = prefill_flops(K, N, M, r) / best / 1e6
            pre.append({"K": K, "N": N, "M": M, "fused_us": round(res["fused"], 1),
                        "stream_us": round(res["stream"], 1), "plain_us": round(res["plain"], 1),
                        "TFLOP_s": round(tfl, 1), "frac_bf16_burst": round(tfl / peaks["bf16_tflops"], 4),
                        "comp_overhead": round(best / res["plain"] - 1, 4),
                        "best_mode": "fused" if res["fused"] <= res["stream"] else "stream"})
            del x, y, ws
        del L0, q, s_, z, A, B, wg
        torch.cuda.empty_cache()
    dec_bytes = sum(decode_bytes(c["K"], c["N"], c["M"], r) for c in dec)
    dec_us = sum(c["us"] for c in dec)
    pre_fl = sum(prefill_flops(c["K"], c["N"], c["M"], r) for c in pre)
    pre_us = sum(min(c["fused_us"], c["stream_us"]) for c in pre)
    return {"workload": "llama70b_g128_r64", "shapes_KxN": [list(t) for t in wl["shapes"]], "rank": r,
            "group_size": Gw, "symmetric": sym,
            "decode": {"GB_s": round(dec_bytes / dec_us / 1e3, 1),
                       "frac_hbm_measured": round(dec_bytes / dec_us / 1e3 / peaks["hbm_gbs"], 4),
                       "comp_overhead": round(dec_us / sum(c["plain_us"] for c in dec) - 1, 4),
                       "l2": "each call on its own weight copy; each shape's copies >= 4x L2", "cases": dec},
            "prefill": {"TFLOP_s": round(pre_fl / pre_us / 1e6, 1),
                        "frac_bf16_burst": round(pre_fl / pre_us / 1e6 / peaks["bf16_tflops"], 4),
                        "cases": pre}}


def run_schedule(args):
    """SLO-constrained chunk selection on the 32-block decoder stack: latency
    tables measured per layer kind, then for several compensator densities and
    inter-token latency targets the chosen prefill chunk, its predicted mixed
    step and the measured one (the stack step at that chunk, CUDA graph)."""
    import torch
    from quantized_gemm_error_gb300 import spear
    from quantized_gemm_error_gb300.scheduler import choose_chunk, measure_curves
    from quantized_gemm_error_gb300.stack import StackStep, build_stack, select_blocks
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    spear.load()
    spear.spear_set_launch_overlap(True)
    D = 32
    choices = [0, 128, 256, 384, 512, 768, 1024, 1536, 2048]
    targets_ms = [8.0, 16.0, 22.0]
    rows = []
    table = None
    for masked in (0, 4, 8):
        ranks = select_blocks(32, masked, 64, seed=0)[1] if masked else [0] * 32
        layers = build_stack(ranks, device, seed=0, recipe="device")
        Ls = [sl.layer for sl in layers]
        t = measure_curves(Ls, [128, 256, 512, 1024, 2048, 2560], [1, 8, 16, 32, 64], device)
        table = t if table is None else {**table, **t}
        for tgt in targets_ms:
            C, pred = choose_chunk(Ls, table, D, choices, tgt * 1e3)
            step = StackStep(layers, max(C + D, 1), D, device, seed=0)
            step.capture()
            name = "prefill" if C > 0 else "decode"
            for _ in range(3):
                step.replay(name)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(step.stream)
            for _ in range(10):
                step.replay(name)
            e1.record(step.stream)
            torch.cuda.synchronize()
            meas = e0.elapsed_time(e1) / 10
            rows.append({"compensated_blocks": masked, "itl_target_ms": tgt, "chunk": C,
                         "predicted_ms": round(pred / 1e3, 3), "measured_ms": round(meas, 3),
                         "slo_met": bool(meas <= tgt)})
            del step
        del layers, Ls
        torch.cuda.empty_cache()
    met = sum(r["slo_met"] for r in rows)
    print(json.dumps({
        "metric": "SLO-constrained chunk selection on the 32-block stack (steps meeting the ITL target)",
        "value": met, "unit": f"of {len(rows)}", "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "llama7b_stack_sym_r64", "decode_tokens": D, "chunk_choices": choices,
                   "launch": "cuda-graph"},
        "decisions": rows, "status": spear.spear_get_device_status()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="host seconds the reference arm aims to spend over all its steps")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decoder-stack and Llama-70B sections of the default line")
    ap.add_argument("--profile-prefill", metavar="K,N,M,MODE,ITERS", default=None,
                    help="run one prefill case ITERS times for a profiler and exit")
    ap.add_argument("--stack", action="store_true",
                    help="time the 32-block decoder stack (mixed prefill step and decode step) instead")
    ap.add_argument("--schedule", action="store_true",
                    help="SLO-constrained chunk selection on the decoder stack: chosen chunks, predicted and "
                         "measured step latencies")
    args = ap.parse_args()
    if args.profile_prefill:
        profile_prefill_case(args.profile_prefill)
        return
    if args.schedule:
        run_schedule(args)
        return
    if args.stack:
        args.warmup = max(3, min(args.warmup, 10))
        args.steps = min(args.steps, 50)
        run_stack(args)
        return
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
