#!/usr/bin/env python3
"""Benchmark of the QSA hot path on one GB300 (or N independent replicas).

One step = one decode window of QSA attention in one call of the library
(qsa_decode_window: q preparation -> block scores -> top-k -> split-KV
attention -> log-sum-exp merge, five chained launches).  The headline workload
is the largest single-GPU decode configuration, the batched long-context
window: 2 slots x 2 rows, 24 q heads / 4 KV heads, head_dim 128, 65,536 and
131,072 filled int8 K/V cells of a 200,000-cell capacity each, 64-cell blocks,
top-k 8,192 cells, one call over both slots' pools.  The metric is decode KV
GB/s: the algorithmic bytes a window must read (every filled K code and scale
for the scores, plus the union of the selected visible cells' K+V codes and
scales for the attention) per second.  L2 (129 MB) is flushed before every
timed step, outside the timed events, by writing a 256 MB buffer and then
reading another 256 MB buffer (so the dirty lines of the write are already
written back when the step starts).

Per-kernel times (and the roofline of the dominant kernel) come from
qsa_decode_window_profile, which runs the same launches one after another with
events between them.  The verify window (5 rows, 32,768 cells, top-k 4,096) is
reported in "decode_verify", the prompt side (2,048 queries against 32,768
cells, 24/4 heads, int8 K/V, on the tensor cores) in "prompt", all on the same
line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain FP64 numpy, the build's
correctness reference) on this machine's host cores, one row of the window per
step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

# The oracle legs run single-threaded per process (the all-core legs use one process per core).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "QSA attn: decode KV GB/s (% HBM peak); prompt int8 TOPS (% peak)"
WORKLOAD = ("decode verify window: 5 rows, 24 q heads / 4 KV heads, head_dim 128, 32,768 int8 K/V cells, "
            "64-cell blocks, top-k 4,096 cells")
LONG_WORKLOAD = ("batched long-context window: 2 slots x 2 rows, 24/4 heads, 65,536 and 131,072 int8 K/V cells, "
                 "top-k 8,192, one call over both slots' pools")
PROMPT_WORKLOAD = "prompt chunk: 2,048 queries at 30,720..32,767 over 32,768 int8 K/V cells, 24/4 heads"
DTYPE = "f16 hi+lo operands on exact int8/4-bit codes, f32 accumulate"
PROMPT_CALLS = 20     # timed prompt calls (independent of --steps)
K8V4_REPEATS = 5      # timed four-call K8V4 prompts
L2_FLUSH_BYTES = 256 << 20
K_ROW, KS_ROW, V_ROW, VS_ROW = 128, 8, 128, 8


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def row_bytes(pool):
    """(K code + scale bytes, V code + scale bytes) of one (cell, KV head) in the pool's layout."""
    k = (K_ROW + KS_ROW) if getattr(pool, "k_bits", 8) == 8 else (K_ROW // 2 + 2 * KS_ROW)
    v = (V_ROW + VS_ROW) if pool.v_bits == 8 else (V_ROW // 2 + 2 * VS_ROW)
    return k, v


def algorithmic_bytes(case, ids, n_sel):
    """(a1 bytes, a3 bytes) of one window: every filled K code + scale once; the union over rows
    of each pool's selected visible cells, K+V codes + scales, once per KV head."""
    a1 = sum(p.n_filled * p.n_kv_heads * row_bytes(p)[0] for p in case.pools)
    a3 = 0
    for pi, pool in enumerate(case.pools):
        cells = set()
        for t in range(case.n_rows):
            if case.row_pool[t] != pi:
                continue
            sel = np.asarray(ids[t][: n_sel[t]])
            cells.update(sel[sel <= case.row_pos[t]].tolist())
        a3 += len(cells) * pool.n_kv_heads * sum(row_bytes(pool))
    return a1, a3


def prompt_flops(case, call):
    """(issued, logical) FLOPs of one prompt call.  Logical: unmasked (query, cell) pairs x q heads x
    2 products x 2 * 128 FLOP.  Issued on the tensor cores: each product three times (the hi.hi, hi.lo
    and lo.hi parts of the fp16 hi + lo operands), six passes in all (the pages' int8 form is the same
    count: three 8-bit planes of the non-code operand per product)."""
    _, n_q, pos0 = call
    pairs = sum(pos0 + i + 1 for i in range(n_q)) * case.n_q_heads
    return pairs * 2 * 128 * 6, pairs * 2 * 2 * 128


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first_sample(self, timeout_s: float = 5.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            time.sleep(0.02)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def slowdown_since(self, n0: int) -> bool:
        """A hardware, hardware-thermal or software-thermal slowdown in the samples taken since sample n0."""
        for ln in self.lines[n0:]:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) == 6 and any(v.lower() == "active" for v in parts[2:5]):
                return True
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary (key "kernel" or "kernel@workload"), if the
    kernel source is unchanged since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)[kernel]
        src = os.path.join(ROOT, "sparse_selection_attention_gb300", "csrc", d["source"])
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return int(d["dram_bytes_per_launch"]) if sha == d["source_sha"] else None
    except Exception:
        return None


# ------------------------------------------------------------------ distributed

def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist
    rank, local = int(os.environ["RANK"]), int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle legs

def oracle_window_seconds(case, budget_s: float):
    """Times the oracle's full decode window repeatedly for about budget_s seconds (one core)."""
    import oracle as O
    reps, t0 = 0, time.perf_counter()
    while True:
        O.decode_window(case)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el / reps, reps


def cpu_baseline(case, builder, bytes_per_window, budget_s=10.0):
    """The oracle's decode window on one host core and on all of them (one process per core, the
    window's rows spread over them, several windows in flight)."""
    from oracle import parallel as OP
    sec, reps = oracle_window_seconds(case, budget_s)
    one = {"value": bytes_per_window / sec / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"full decode window (all 4 steps, {case.n_rows} rows) x {reps}, {sec * 1e3:.0f} ms each, "
                     "FP64 numpy, one thread"}
    n = OP.workers()
    runner = OP.WindowRunner(builder, {}, n)
    try:
        runner.run(1)   # workers started and holding the case
        n_win = max(1, int(round(budget_s / sec * n / 2)))
        t0 = time.perf_counter()
        runner.run(n_win)
        el = time.perf_counter() - t0
    finally:
        runner.close()
    return {"value": bytes_per_window * n_win / el / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "nproc": os.cpu_count(),
            "sample": f"{n_win} full decode windows, their rows spread over {n} processes (one per core), "
                      f"{el:.1f} s, FP64 numpy",
            "single_core": one}


def prompt_cpu_baseline(pcase, call, flops_issued, budget_s=6.0):
    """The oracle's prompt attention on one core (random 16-row blocks, all heads, for about budget_s)
    and on all cores (every row of the call)."""
    import oracle as O
    from oracle import parallel as OP
    rng = np.random.default_rng(0)
    i0, n_q, pos0 = call
    rows, t0 = [], time.perf_counter()
    q = pcase.q[i0:i0 + n_q]
    while time.perf_counter() - t0 < budget_s:
        r0 = int(rng.integers(0, n_q - 16))
        O.prompt_attention(pcase.pool, q, pos0, rows=list(range(r0, r0 + 16)))
        rows.extend(range(r0, r0 + 16))
    el = time.perf_counter() - t0
    total_pairs = sum(pos0 + i + 1 for i in range(n_q)) * pcase.n_q_heads
    per_pair = flops_issued / total_pairs
    pairs = sum(pos0 + r + 1 for r in rows) * pcase.n_q_heads
    one = {"value": pairs * per_pair / el / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
           "sample": f"{len(rows)} query rows of the 2,048-query call in 16-row blocks, all heads, FP64 numpy"}
    n = OP.workers()
    rows_all = list(range(n_q - 8 * n, n_q))   # 8 rows per process, at the call's longest contexts
    t0 = time.perf_counter()
    OP.prompt_call("prompt_int8", {}, 0, row_block=8, rows=rows_all)
    el = time.perf_counter() - t0
    pairs_all = sum(pos0 + r + 1 for r in rows_all) * pcase.n_q_heads
    return {"value": pairs_all * per_pair / el / 1e12, "unit": "TFLOP/s", "cores": n, "kind": "oracle",
            "nproc": os.cpu_count(),
            "sample": f"the call's last {len(rows_all)} query rows, all heads, in 8-row tasks over {n} processes "
                      f"(one per core), {el:.1f} s including the workers' start-up, FP64 numpy",
            "single_core": one}


# ------------------------------------------------------------------ our arm

def gpu_sleep(us: float = 400.0):
    """Keeps the GPU busy for about `us` microseconds (outside any timed event)."""
    import torch
    torch.cuda._sleep(int(us * 2.1e3))


def window_of(case, dev):
    import torch

    import sparse_selection_attention_gb300 as qsa
    pools = [qsa.DevicePool.upload(p, dev) for p in case.pools]
    win = qsa.DecodeWindow(pools, case.row_pool, case.n_q_heads, case.block_cells, case.k_cells, case.chunk_cells,
                           n_chunks=case.n_chunks, max_blocks=case.max_blocks, device=dev)
    return win, torch.from_numpy(case.q).to(dev), torch.from_numpy(case.row_pos).to(dev)


KERNELS = ["q_prep", "block_scores", "topk", "split_attn", "merge"]


def workload_config(case, a1, a3, workload):
    """The workload part of the JSON line's config, the same for both arms."""
    return {"workload": workload, "rows": case.n_rows, "q_heads": case.n_q_heads, "kv_heads": case.pools[0].n_kv_heads,
            "cells": [p.n_filled for p in case.pools], "k_cells": case.k_cells, "block_cells": case.block_cells,
            "bytes_per_step": a1 + a3, "scores_bytes": a1, "attention_union_bytes": a3}
K8V4_WORKLOAD = ("large prompt with mixed KV: 8,192 queries at 122,880..131,071 over 131,072 cells, 32/8 heads, "
                 "int8 K / 4-bit V, four calls of 2,048 queries in one stream")


def run_kv_append(dev, stream, flush_l2, hbm_peak, ws):
    """qsa_kv_append of (a) one 2,048-cell prompt chunk into the int8 prompt pool's shape (4 KV heads)
    and (b) 32,768 cells x 8 KV heads into a K8V4 pool: algorithmic bytes per (cell, KV head) are the
    fp32 K and V rows read (1,024 B) plus the codes and scales written (136 B for int8 K; 136 B for
    int8 V, 80 B for 4-bit V)."""
    import torch

    import sparse_selection_attention_gb300 as qsa
    res = {}
    for name, n, Hkv, v_bits, cap in (("prompt_chunk_2048x4_int8", 2048, 4, 8, 32768),
                                      ("cells_32768x8_k8v4", 32768, 8, 4, 32768)):
        rng = np.random.default_rng(n + Hkv)
        pool = qsa.DevicePool.upload(W.make_pool(rng, capacity=cap, n_filled=0, n_kv_heads=Hkv, page_cells=256,
                                                 v_bits=v_bits), dev)
        k = torch.randn((n, Hkv, 128), device=dev)
        v = torch.randn((n, Hkv, 128), device=dev)
        for _ in range(3):
            qsa.kv_append(pool, k, v, 0)
        torch.cuda.synchronize()
        ts = []
        for _ in range(10):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            qsa.kv_append(pool, k, v, 0)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        us = max_over_ranks(float(np.mean(ts)), ws) * 1e3
        nbytes = n * Hkv * (1024 + 136 + (136 if v_bits == 8 else 80))
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us": us, "algorithmic_bytes": nbytes, "GB/s": gbs * ws, "frac_hbm": gbs / hbm_peak}
        if name == "cells_32768x8_k8v4":
            res[name]["traffic"] = kernel_traffic("kv_append")   # DRAM bytes per launch (ncu), or None
    return res


def run_prompt_k8v4(dev, stream, flush_l2, tc_peak, ws):
    """The four 2,048-query calls of the K8V4 prompt, one after another on one stream, timed together."""
    import torch

    import sparse_selection_attention_gb300 as qsa
    case = W.prompt_k8v4()
    pool = qsa.DevicePool.upload(case.pool, dev)
    q = torch.from_numpy(case.q).to(dev)
    n = max(c[1] for c in case.calls)
    out = torch.empty((n, case.n_q_heads, 128), device=dev)
    lse = torch.empty((n, case.n_q_heads), device=dev)
    need = max(qsa.prompt_scratch_bytes(pool, c[1], c[2], case.n_q_heads) for c in case.calls)
    scratch = torch.empty(max(1, need), dtype=torch.uint8, device=dev)

    def chunked():
        for i0, nq, pos0 in case.calls:
            qsa.prompt_attn(pool, q[i0:i0 + nq], pos0, out[:nq], lse[:nq], scratch=scratch)
    chunked()
    torch.cuda.synchronize()
    times = []
    for _ in range(K8V4_REPEATS):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        chunked()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    if qsa.get_device_error() != 0:
        raise RuntimeError("prompt kernel reported a device error")
    ms = max_over_ranks(float(np.mean(times)), ws)
    issued = sum(prompt_flops(case, c)[0] for c in case.calls)
    logical = sum(prompt_flops(case, c)[1] for c in case.calls)
    ach = issued / (ms * 1e-3) / 1e12
    return {"workload": K8V4_WORKLOAD, "ms_per_prompt": ms, "value": ach * ws, "unit": "TFLOP/s",
            "logical_TFLOP/s": logical / (ms * 1e-3) / 1e12 * ws, "frac_of_tensor_peak": ach / tc_peak,
            "scratch_bytes": need}


def run_ours(args):
    import torch

    import sparse_selection_attention_gb300 as qsa  # noqa: F401  (fails loudly without the CUDA library)

    rank, ws, local = dist_init()
    if args.gpus != ws:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but {ws} process(es) were launched (one per GPU: run "
                         f"N > 1 under torchrun with --nproc-per-node N)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, peak_src = peaks()

    builder = "verify_window" if args.case == "verify" else "batched_long_context"
    case = getattr(W, builder)()
    win, q, row_pos = window_of(case, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        """Writes 256 MB (evicts L2), then reads another 256 MB so that the dirty lines are written
        back before the timed work starts (it then finds a cold, clean L2)."""
        flush.zero_()
        clean.sum()
    stream = torch.cuda.current_stream(dev)

    clocks = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        win.run_window(q, row_pos)
    torch.cuda.synchronize()
    clocks.wait_first_sample()
    ids = win.ids.cpu().numpy()
    n_sel = win.n_sel.cpu().numpy()
    a1, a3 = algorithmic_bytes(case, [ids[t] for t in range(case.n_rows)], n_sel)
    bytes_step = a1 + a3

    # ---- device-timed steps: one qsa_decode_window call each, events on the launching stream
    # A run whose clock samples show a hardware or thermal slowdown is taken once more.
    K = args.steps
    remeasured = False
    for attempt in range(2):
        n0 = len(clocks.lines)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        barrier(ws)
        torch.cuda.synchronize()
        for k in range(K):
            flush_l2()
            gpu_sleep()   # the GPU idles here, outside the events, while the CPU enqueues the step
            ev[k][0].record(stream)
            win.run_window(q, row_pos)
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        time.sleep(0.05)   # the sampler's last samples of the timed region
        slow = max_over_ranks(1.0 if clocks.slowdown_since(n0) else 0.0, ws) > 0.0   # the ranks decide together
        if attempt == 1 or not slow:
            break
        remeasured = True
    step_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    step_ms = max_over_ranks(step_ms, ws)
    value = bytes_step * ws / (step_ms * 1e-3) / 1e9

    # ---- the same call replayed from a CUDA graph (how a serving loop issues a decode window; the
    # pages' kernel timings are graph replays): one submission for the five chained launches
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        win.run_window(q, row_pos)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        flush_l2()
        gpu_sleep()
        gev[k][0].record(stream)
        graph.replay()
        gev[k][1].record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in gev])), ws)
    graph_replay = {"ms_per_step": graph_ms, "value": bytes_step * ws / (graph_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "gpu_launches": 5 * K}

    # ---- per-kernel times: the same launches without overlap, events between them
    P = max(5, min(50, K // 4))
    per = []
    for _ in range(P):
        flush_l2()
        gpu_sleep()
        per.append(win.run_window_profile(q, row_pos))
    kern_us = np.mean(np.array(per), axis=0)
    byte_of = {"block_scores": a1, "split_attn": a3}
    kernels = {}
    for j, n in enumerate(KERNELS):
        d = {"us": float(kern_us[j]), "share": float(kern_us[j] / kern_us.sum())}
        if n in byte_of:
            d["algorithmic_bytes"] = byte_of[n]
            d["GB/s"] = byte_of[n] / (kern_us[j] * 1e-6) / 1e9
            d["frac_hbm"] = d["GB/s"] / hbm_peak
        kernels[n] = d
    dom = max(byte_of, key=lambda n: kern_us[KERNELS.index(n)])
    ach = byte_of[dom] / (kern_us[KERNELS.index(dom)] * 1e-6) / 1e9
    roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                "frac": ach / hbm_peak, "peak_source": f"{peak_src} hbm_gbs (burst copy; kernel timed alone)",
                "algorithmic_bytes": byte_of[dom], "traffic": kernel_traffic(f"{dom}@{args.case}"),
                "timing": "qsa_decode_window_profile: CUDA events around the launch, no overlap with its neighbours"}

    # ---- the four separate calls (qsa_block_scores, qsa_topk, qsa_decode_attn, qsa_attn_merge), for context
    sep = []
    for _ in range(P):
        flush_l2()
        gpu_sleep()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        win.run(q, row_pos)
        b.record(stream)
        torch.cuda.synchronize()
        sep.append(a.elapsed_time(b))

    # ---- end to end through the public API with page-locked host buffers: qsa_decode_window_host reads
    # the step's inputs (q and the row positions) from host memory into its workspace and writes its
    # results (out and lse) back there, across the host link, inside the timed region
    q_h = torch.from_numpy(np.ascontiguousarray(case.q)).pin_memory()
    pos_h = torch.from_numpy(np.ascontiguousarray(case.row_pos.astype(np.int32))).pin_memory()
    out_h = torch.empty(tuple(win.out.shape), dtype=torch.float32).pin_memory()
    lse_h = torch.empty(tuple(win.lse.shape), dtype=torch.float32).pin_memory()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    for k in range(K):
        flush_l2()
        gpu_sleep()   # outside the events: the host enqueues the step while the GPU idles here
        e2e_ev[k][0].record(stream)
        win.run_window_host(q_h, pos_h, out_h, lse_h)
        e2e_ev[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in e2e_ev]))
    e2e_ms = max_over_ranks(e2e_ms, ws)
    h2d = q_h.numel() * 4 + pos_h.numel() * 4
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    win.run_window(q, row_pos)
    torch.cuda.synchronize()
    if not (torch.equal(out_h, win.out.cpu()) and torch.equal(lse_h, win.lse.cpu())):
        raise RuntimeError("end-to-end results differ from the device's")

    # ---- the other decode window (secondary): the verify window under the long-context headline
    decode_other, other_key = None, "decode_verify" if args.case == "long" else "decode_long"
    if not args.no_long:
        ocase = W.verify_window() if args.case == "long" else W.batched_long_context()
        owin, oq, opos = window_of(ocase, dev)
        for _ in range(3):
            owin.run_window(oq, opos)
        torch.cuda.synchronize()
        oids = owin.ids.cpu().numpy()
        osel = owin.n_sel.cpu().numpy()
        o1, o3 = algorithmic_bytes(ocase, [oids[t] for t in range(ocase.n_rows)], osel)
        ot = []
        for _ in range(P):
            flush_l2()
            gpu_sleep()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            owin.run_window(oq, opos)
            b.record(stream)
            torch.cuda.synchronize()
            ot.append(a.elapsed_time(b))
        oper = []
        for _ in range(5):
            flush_l2()
            gpu_sleep()
            oper.append(owin.run_window_profile(oq, opos))
        oper = np.mean(np.array(oper), axis=0)
        oms = max_over_ranks(float(np.mean(ot)), ws)
        decode_other = {"workload": WORKLOAD if args.case == "long" else LONG_WORKLOAD, "ms_per_step": oms,
                        "value": (o1 + o3) * ws / (oms * 1e-3) / 1e9, "unit": "GB/s",
                        "frac_of_hbm_peak": (o1 + o3) / (oms * 1e-3) / 1e9 / hbm_peak,
                        "bytes_per_step": o1 + o3, "scores_bytes": o1, "attention_union_bytes": o3,
                        "kernels_us": dict(zip(KERNELS, [float(x) for x in oper]))}

    # ---- windows whose pools keep block summaries (qsa_pool.k_sums, built outside the timing): the same
    # scores from 512 bytes per 64 cells and KV head instead of the codes and scales
    def time_with_block_sums(bcase, workload):
        spools = [qsa.DevicePool.upload(p, dev).keep_block_sums() for p in bcase.pools]
        swin = qsa.DecodeWindow(spools, bcase.row_pool, bcase.n_q_heads, bcase.block_cells, bcase.k_cells,
                                bcase.chunk_cells, n_chunks=bcase.n_chunks, max_blocks=bcase.max_blocks, device=dev)
        sq, spos = torch.from_numpy(bcase.q).to(dev), torch.from_numpy(bcase.row_pos).to(dev)
        for _ in range(3):
            swin.run_window(sq, spos)
        torch.cuda.synchronize()
        sids, ssel = swin.ids.cpu().numpy(), swin.n_sel.cpu().numpy()
        _, s3 = algorithmic_bytes(bcase, [sids[t] for t in range(bcase.n_rows)], ssel)
        s1 = sum((p.n_filled + 63) // 64 * p.n_kv_heads * 512 for p in bcase.pools)
        st = []
        for _ in range(P):
            flush_l2()
            gpu_sleep()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            swin.run_window(sq, spos)
            b.record(stream)
            torch.cuda.synchronize()
            st.append(a.elapsed_time(b))
        sper = []
        for _ in range(5):
            flush_l2()
            gpu_sleep()
            sper.append(swin.run_window_profile(sq, spos))
        sms = max_over_ranks(float(np.mean(st)), ws)
        return {"workload": workload + ", blocks scored from the pools' block summaries", "ms_per_step": sms,
                "value": (s1 + s3) * ws / (sms * 1e-3) / 1e9, "unit": "GB/s", "bytes_per_step": s1 + s3,
                "summary_bytes": s1, "attention_union_bytes": s3,
                "kernels_us": dict(zip(KERNELS, [float(x) for x in np.mean(np.array(sper), axis=0)]))}

    decode_sums = decode_other_sums = None
    if not args.no_long:
        decode_sums = time_with_block_sums(getattr(W, builder)(), WORKLOAD if args.case == "verify" else LONG_WORKLOAD)
        decode_sums["speedup_vs_headline"] = step_ms / decode_sums["ms_per_step"]
        decode_other_sums = time_with_block_sums(W.verify_window() if args.case == "long" else W.batched_long_context(),
                                                 WORKLOAD if args.case == "long" else LONG_WORKLOAD)

    # ---- prompt side
    prompt = None
    if not args.no_prompt:
        import sparse_selection_attention_gb300 as qsa
        pcase = W.prompt_int8()
        call = pcase.calls[0]
        ppool = qsa.DevicePool.upload(pcase.pool, dev)
        pq = torch.from_numpy(pcase.q).to(dev)
        pout = torch.empty((call[1], pcase.n_q_heads, 128), device=dev)
        plse = torch.empty((call[1], pcase.n_q_heads), device=dev)
        pscratch = torch.empty(max(1, qsa.prompt_scratch_bytes(ppool, call[1], call[2], pcase.n_q_heads)), dtype=torch.uint8,
                               device=dev)
        for _ in range(2):
            qsa.prompt_attn(ppool, pq, call[2], pout, plse, scratch=pscratch)
        torch.cuda.synchronize()
        PP = PROMPT_CALLS
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(PP)]
        for k in range(PP):
            flush_l2()
            pev[k][0].record(stream)
            qsa.prompt_attn(ppool, pq, call[2], pout, plse, scratch=pscratch)
            pev[k][1].record(stream)
        torch.cuda.synchronize()
        if qsa.get_device_error() != 0:
            raise RuntimeError("prompt kernel reported a device error")
        p_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in pev])), ws)
        issued, logical = prompt_flops(pcase, call)
        ach_p = issued / (p_ms * 1e-3) / 1e12
        prompt = {"workload": PROMPT_WORKLOAD, "ms_per_call": p_ms, "value": ach_p * ws, "unit": "TFLOP/s",
                  "logical_TFLOP/s": logical / (p_ms * 1e-3) / 1e12 * ws, "dtype": DTYPE, "calls_timed": PP,
                  "roofline": {"kernel": "prompt_attn", "bound": "tensor", "achieved": ach_p, "peak": tc_peak,
                               "unit": "TFLOP/s", "frac": ach_p / tc_peak,
                               "peak_source": f"{peak_src} bf16_tflops (fp16 dense rate = bf16)",
                               "traffic": kernel_traffic("prompt_attn")}}
        # The metric's prompt denominator is the dense int8 rate.  tcgen05 has no int8 kind on this GPU,
        # so that rate is the mma.sync s8 one; the pages' form issues the same six passes per product
        # pair as int8 operations that this path issues as fp16 ones.
        i8_rate = qsa.measure_tc_rate(qsa.QSA_TC_KIND_I8, 50) / 1e12
        f16_rate = qsa.measure_tc_rate(qsa.QSA_TC_KIND_F16, 10000) / 1e12
        prompt["int8"] = {"achieved_TOPS": ach_p, "peak_TOPS": i8_rate, "frac": ach_p / i8_rate,
                          "peak_source": "measured in this run (qsa_measure_tc_rate: mma.sync m16n8k32 s8, 16 warps "
                                         "per SM; tcgen05.mma has no kind::i8 on sm_103a)",
                          "note": "issued operations counted as the pages' int8 form counts them (3 planes x 2 "
                                  "products); this path issues them as fp16 hi/lo products"}
        prompt["f16_tcgen05_probe_TFLOPS"] = f16_rate
        if rank == 0 and ws == 1 and not args.no_cpu_baseline:
            prompt["cpu_baseline"] = prompt_cpu_baseline(pcase, call, issued)
        del pscratch
        if not args.no_k8v4:
            prompt["k8v4"] = run_prompt_k8v4(dev, stream, flush_l2, tc_peak, ws)

    kv_append = None if args.no_append else run_kv_append(dev, stream, flush_l2, hbm_peak, ws)
    decode_tiny = None
    if not args.no_long:
        tcase = W.tiny_dense_decode()
        twin, tq, tpos = window_of(tcase, dev)
        for _ in range(3):
            twin.run_window(tq, tpos)
        torch.cuda.synchronize()
        tt = []
        for _ in range(P):
            flush_l2()
            gpu_sleep()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            twin.run_window(tq, tpos)
            b.record(stream)
            torch.cuda.synchronize()
            tt.append(a.elapsed_time(b))
        decode_tiny = {"workload": "tiny dense decode: 1 row, 2 q heads / 1 KV head, 1,024 int8 K/V cells, top-k = all "
                                   "cells (latency-bound: microseconds per call)",
                       "us_per_call": max_over_ranks(float(np.mean(tt)), ws) * 1e3}
    decode_q4_0 = None
    if not args.no_long:
        qcase = W.decode_case(name="q4_0 verify window", seed=11, fills=[32768], capacity=32768, rows_per_slot=5,
                              n_q_heads=24, n_kv_heads=4, k_cells=4096, chunk_cells=64, v_bits=4, k_bits=4,
                              bias_prob=0.05)
        qwin, qq, qpos = window_of(qcase, dev)
        for _ in range(3):
            qwin.run_window(qq, qpos)
        torch.cuda.synchronize()
        qids, qsel = qwin.ids.cpu().numpy(), qwin.n_sel.cpu().numpy()
        q1, q3 = algorithmic_bytes(qcase, [qids[t] for t in range(qcase.n_rows)], qsel)
        qt = []
        for _ in range(P):
            flush_l2()
            gpu_sleep()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            qwin.run_window(qq, qpos)
            b.record(stream)
            torch.cuda.synchronize()
            qt.append(a.elapsed_time(b))
        qms = max_over_ranks(float(np.mean(qt)), ws)
        decode_q4_0 = {"workload": "decode verify window in the q4_0 layout (4-bit K and V, 32-dim scale groups): 5 rows, "
                                   "24/4 heads, 32,768 cells, top-k 4,096", "ms_per_step": qms,
                       "value": (q1 + q3) * ws / (qms * 1e-3) / 1e9, "unit": "GB/s", "bytes_per_step": q1 + q3}

    clocks.__exit__()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": {**workload_config(case, a1, a3, WORKLOAD if args.case == "verify" else LONG_WORKLOAD),
                   "call": "qsa_decode_window (5 launches chained by programmatic dependent launch)",
                   "l2": "flushed before every timed step, outside the events: 256 MB write, then 256 MB read",
                   "parallelism": f"{ws} independent replica(s)" if ws > 1 else "1 GPU"},
        "frac_of_hbm_peak": value / ws / hbm_peak,
        "roofline": roofline,
        "kernels": kernels,
        "separate_calls_ms": float(np.mean(sep)),
        "graph_replay": graph_replay,
        "kv_append": kv_append,
        "decode_q4_0": decode_q4_0,
        "decode_tiny": decode_tiny,
        "e2e": {"value": bytes_step * ws / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "call": "qsa_decode_window_host: q and row positions staged from page-locked host memory by the "
                        "window's first launch, out and lse written back to host memory by its merge"},
        "gpu_launches": 5 * K,
        "clocks": dict(clocks.summary(), remeasured_after_slowdown=remeasured),
        other_key: decode_other,
        "decode_block_sums": decode_sums,
        other_key + "_block_sums": decode_other_sums,
        "prompt": prompt,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, builder, bytes_step)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as the reference arm, on this arm's workload: step k computes row k mod R of the
    window (its pool's block scores, full-sort top-k, chunk partials, merge) on one host core; the
    window time is the sum over rows of each row's mean step time."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as O
    case = W.verify_window() if args.case == "verify" else W.batched_long_context()
    res = O.decode_window(case)
    a1, a3 = algorithmic_bytes(case, res["ids"], res["n_sel"])
    bytes_step = a1 + a3
    R = case.n_rows

    def row(t):
        pool = case.pools[case.row_pool[t]]
        s = O.block_scores(pool, case.q[[t]], case.block_cells)[0]
        sel, _ = O.topk_select(s.astype(np.float32), pool.n_filled, case.block_cells, case.k_cells)
        m, l, o = O.chunk_partials(pool, case.q[t], int(case.row_pos[t]), sel, case.chunk_cells, case.n_chunks)
        O.merge_partials(m, l, o)
    for k in range(args.warmup):
        row(k % R)
    per_row = [[] for _ in range(R)]
    for k in range(args.steps):
        t0 = time.perf_counter()
        row(k % R)
        per_row[k % R].append(time.perf_counter() - t0)
    mean_row = [np.mean(x) if x else np.mean([y for z in per_row for y in z]) for x in per_row]
    ms = float(np.sum(mean_row)) * 1e3   # one whole window
    value = bytes_step / (ms * 1e-3) / 1e9
    step_ms = float(np.mean([y for z in per_row for y in z])) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "ms_per_window": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": {**workload_config(case, a1, a3, WORKLOAD if args.case == "verify" else LONG_WORKLOAD),
                   "call": "the oracle's decode chain, one row of the window per step (oracle/qsa_oracle.py)",
                   "parallelism": "1 host core"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} rows of the window ({R} rows), one per step: block scores, full-sort "
                                   "top-k, chunk partials, merge; FP64 numpy, one thread"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prompt", action="store_true")
    ap.add_argument("--no-k8v4", action="store_true", help="skip the K8V4 prompt (four calls over 131,072 cells)")
    ap.add_argument("--no-append", action="store_true", help="skip the quantise-on-append measurement")
    ap.add_argument("--no-long", "--no-secondary", dest="no_long", action="store_true",
                    help="skip the secondary decode workloads (the other window, tiny, q4_0)")
    ap.add_argument("--case", choices=["verify", "long"], default="long",
                    help="decode workload of the timed step (the batched long-context window is the headline)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
