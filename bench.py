#!/usr/bin/env python3
"""Benchmark: one Muon step with Gram Newton-Schulz over a batch of 24 bf16 matrices
1024 x 4096 (dense-MLP projections, alpha = 4), i.e. momentum EMA (mu = 0.95), Frobenius
normalisation, Gram NS (T = 5, fixed quintic, restart after iteration 2) and the weight
update (lr = 0.02), all in libgns kernels on one GPU per process.

Prints ONE JSON line (rank 0). `value` is whole-job matrices/s with inputs resident in HBM;
`e2e` is the same metric with the gradient copied in from pinned host memory and the
updated weights copied back every step; `roofline` rates the dominant kernel (the
tcgen05 GEMM) from CUDA events recorded around each of its launches in an instrumented
repeat of the timed loop; `cpu_baseline` times the fp64 CPU oracle on a bounded sample.

`--impl reference` times the CPU oracle itself (the only reference there is) with the same
metric and unit, each step one matrix of the workload.

Multi-GPU (torchrun): replicas only — every rank runs the same workload on its own GPU;
there is no data-path collective. Timing is barrier-bracketed and the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Gram-NS orthogonalized matrices/s and TFLOP/s vs BF16 tensor peak (α=4, T=5)"
UNIT = "matrices/s"
COUNT, ROWS, COLS = 24, 1024, 4096
LR, MU = 0.02, 0.95
WORKLOAD = "muon_step bf16 24 x 1024x4096 (alpha=4): momentum 0.95, Gram NS T=5 fixed quintic restart@2, lr 0.02"


def alg_flops_per_matrix(n=ROWS, m=COLS):
    """(14 + 6 alpha) n^3: Gram NS with one restart (Dion3 sec. 4.1 + 4.2), symmetric
    products counted as n^3 (sec. 2.3)."""
    alpha = m / n
    return (14 + 6 * alpha) * n ** 3


def std_flops_per_matrix(n, m, T=5):
    """T (3 alpha + 1) n^3: standard Newton-Schulz with symmetric products (Dion3 sec. 2.3)."""
    return T * (3 * m / n + 1) * n ** 3


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the GEMM kernel
# on this workload, from an ncu capture of `bench.py --metric-only`, keyed by the sha256
# prefix of the kernel sources it was taken on with comments and blank lines removed (a
# comment edit leaves the kernel unchanged): reported only while that code is unchanged
# (null otherwise), never measured inside this run.
GEMM_TRAFFIC = {"e317f1a863859d40": 2.297286e9}


def gemm_source_hash():
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "common.cuh"):
        src = open(os.path.join(ROOT, "matrix_orthogonalizing_optimizer_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("\n".join(line.rstrip() for line in src.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def gemm_traffic():
    return GEMM_TRAFFIC.get(gemm_source_hash())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# ---------------------------------------------------------------------------------------
# replicas: every rank runs the whole workload on its own GPU; no data-path collective

def max_over_ranks_of(dist, x, device="cpu"):
    """Largest value of x over the ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, ms_per_step_max):
    """Units all ranks processed per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_per_step_max / 1000.0)


# ---------------------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2] if sm_sorted else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------------------
# CPU oracle timing

def time_oracle(n_matrices, seed=1):
    import numpy as np
    from matrix_orthogonalizing_optimizer_gb300 import inputs
    from oracle import muon as omuon
    s = 1.0 / np.sqrt(COLS)
    mats = []
    for i in range(n_matrices):
        W = inputs.round_to_bf16_bits(inputs.gaussian(seed, (ROWS, COLS), s, stream=10 * i))
        G = inputs.round_to_bf16_bits(inputs.gaussian(seed, (ROWS, COLS), s, stream=10 * i + 1))
        M = inputs.round_to_bf16_bits(inputs.gaussian(seed, (ROWS, COLS), s, stream=10 * i + 2))
        mats.append((W, G, M))
    t0 = time.perf_counter()
    for (W, G, M) in mats:
        omuon.muon_step(W, G, M, lr=LR, mu=MU)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def bench_config(world):
    """The workload both arms name in their line's config."""
    return {"workload": WORKLOAD, "matrices": COUNT, "rows": ROWS, "cols": COLS,
            "l2": "inputs larger than L2 (W, G, M: 604 MB per rank)", "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        time_oracle(1)
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle(1)
    v = args.steps / total
    sample = "1 of the 24 matrices per step (fp64 numpy oracle: momentum, Gram NS restart@2, update)"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------
# GPU arm

def run_ours(args, rank, world, dist):
    import ctypes

    import torch

    import matrix_orthogonalizing_optimizer_gb300 as gns
    from matrix_orthogonalizing_optimizer_gb300 import _lib

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = _lib.load()

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    s = 1.0 / COLS ** 0.5

    def randn():
        return (torch.randn((COUNT, ROWS, COLS), generator=gen, device=dev, dtype=torch.float32) * s).to(torch.bfloat16)

    W = randn()
    M = torch.zeros((COUNT, ROWS, COLS), dtype=torch.bfloat16, device=dev)
    G1, G2, G = randn(), randn(), randn()
    ns = gns.NsParams()
    ws = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_MUON_STEP, M, ns), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def time_orth(X, fn, op, flops):
        """One batched orthogonalization call (warm-up, then 3 timed calls): call time and the
        GEMM launches' time from the library's event hooks."""
        Xo = torch.empty_like(X)
        ws_m = gns.alloc_workspace(gns.workspace_size(op, X, ns), dev)
        # the bench's status word: the calls run back to back without a host synchronisation
        # after each (the word is checked once the timed calls are done)
        fn(X, outs=[Xo], ns=ns, workspace=ws_m, stream=stream, status=status)
        torch.cuda.synchronize()
        reps = 3
        evm = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
        for e in evm:
            e.record(stream)
        hm = (ctypes.c_void_p * (2 * reps))(*[ctypes.c_void_p(e.cuda_event) for e in evm])
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lib.gns_profile_set(hm, reps)
        a.record(stream)
        for _ in range(reps):
            fn(X, outs=[Xo], ns=ns, workspace=ws_m, stream=stream, status=status)
        b.record(stream)
        torch.cuda.synchronize()
        gns.check_status(status, what="bench orthogonalization")
        lib.gns_profile_set(None, 0)
        call_ms = a.elapsed_time(b) / reps
        g_ms = sum(evm[2 * i].elapsed_time(evm[2 * i + 1]) for i in range(reps)) / reps
        del Xo, ws_m
        torch.cuda.empty_cache()
        tf = flops / (g_ms / 1000.0) / 1e12
        return {"ms_per_call": call_ms, "matrices_per_s": X.shape[0] / (call_ms / 1000.0), "gemm_ms": g_ms,
                "gemm_tflops": tf, "gemm_frac_of_burst_peak": tf / load_peaks()[0],
                "gemm_frac_of_sustained_peak": tf / load_peaks()[1]}

    def small_batches():
        """Groups of small matrices: the on-chip chain kernel (one CTA per matrix, oriented X
        at most 128 x 512) where it applies, else the batched tile path; for chain-kernel
        shapes the tile path is timed beside it (GNS_CHAIN_SMALL=0)."""
        res = {}
        for (count, n, m) in [(2048, 128, 512), (4096, 64, 256), (8192, 32, 128), (512, 256, 1024), (96, 512, 2048)]:
            X = (torch.randn((count, n, m), generator=gen, device=dev, dtype=torch.float32) / m ** 0.5).to(
                torch.bfloat16)
            r = time_orth(X, gns.gram_ns_batched, _lib.GNS_OP_GRAM_NS, count * alg_flops_per_matrix(n, m))
            std = time_orth(X, gns.ns_standard_batched, _lib.GNS_OP_NS_STANDARD, count * std_flops_per_matrix(n, m))
            r["standard_ns_ms_per_call"] = std["ms_per_call"]
            r["gram_vs_standard_speedup"] = std["ms_per_call"] / r["ms_per_call"]
            chain = n <= 128 and m <= 512
            pack = 4 if n <= 32 else 2 if n <= 64 else 1
            # the library's tile plan: 1-CTA 128 x 128 tiles for products of at most 256 rows and
            # for n <= 1024 batches whose largest symmetric stage has at most 48 pair tiles
            t = (n + 255) // 256
            one_cta = n <= 256 or (n <= 1024 and count * t * (t + 1) // 2 <= 48)
            r["path"] = (f"on-chip chain kernel, {pack} matrices per CTA chain" if chain else
                         "batched tiles, 1-CTA 128 x 128" if one_cta else "batched tiles, 2-CTA 256 x 256")
            if chain:
                os.environ["GNS_CHAIN_SMALL"] = "0"
                try:
                    tg = time_orth(X, gns.gram_ns_batched, _lib.GNS_OP_GRAM_NS, count * alg_flops_per_matrix(n, m))
                    ts = time_orth(X, gns.ns_standard_batched, _lib.GNS_OP_NS_STANDARD,
                                   count * std_flops_per_matrix(n, m))
                finally:
                    del os.environ["GNS_CHAIN_SMALL"]
                r["tile_path"] = {"gram_ns_ms_per_call": tg["ms_per_call"], "standard_ns_ms_per_call": ts["ms_per_call"],
                                  "chain_speedup_gram": tg["ms_per_call"] / r["ms_per_call"],
                                  "chain_speedup_standard": ts["ms_per_call"] / std["ms_per_call"]}
            res[f"{count}x{n}x{m}"] = r
            del X
            torch.cuda.empty_cache()
        # several small shape groups in one call (one chain-kernel launch carries them all)
        # against one call per group
        shapes = [(1024, 128, 512), (600, 96, 384), (300, 64, 256), (150, 128, 256), (77, 112, 448)]
        Xs = [(torch.randn((c, n, m), generator=gen, device=dev, dtype=torch.float32) / m ** 0.5).to(torch.bfloat16)
              for (c, n, m) in shapes]
        Os = [torch.empty_like(X) for X in Xs]
        ws_all = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_GRAM_NS, Xs, ns), dev)

        def one_call():
            gns.gram_ns_batched(Xs, outs=Os, ns=ns, workspace=ws_all, stream=stream, status=status)

        def per_group():
            for X, O in zip(Xs, Os):
                gns.gram_ns_batched(X, outs=[O], ns=ns, workspace=ws_all, stream=stream, status=status)

        def t_call(fn, reps=5):
            fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps
        t1, tg = t_call(one_call), t_call(per_group)
        gns.check_status(status, what="bench mixed groups")
        fl = sum(c * alg_flops_per_matrix(n, m) for (c, n, m) in shapes)
        res["mixed_groups_one_call"] = {
            "groups": [f"{c}x{n}x{m}" for (c, n, m) in shapes], "matrices": sum(c for c, _, _ in shapes),
            "one_call_ms": t1, "one_call_per_group_ms": tg, "speedup": tg / t1,
            "tflops_one_call": fl / (t1 / 1000.0) / 1e12,
            "what": "Gram NS of five small shape groups: one call (one chain-kernel launch) vs one call per group"}
        del Xs, Os, ws_all
        torch.cuda.empty_cache()
        return res

    if args.small_only:
        # the small-matrix section alone (for profiling the chain kernel): one JSON line
        if rank == 0:
            print(json.dumps({"small_matrices": small_batches(),
                              "note": "--small-only: the small-matrix section alone, not a bench line"}), flush=True)
        return 0


    def step(g):
        gns.muon_step(W, g, M, lr=LR, momentum=MU, ns=ns, workspace=ws, status=status, stream=stream)

    # the configuration's two earlier synthetic gradient steps, then warm-up on G
    step(G1)
    step(G2)
    for _ in range(args.warmup):
        step(G)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(x):
        return max_over_ranks_of(dist, x, dev)

    # ---- timed region: inputs resident in HBM ----
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lib.gns_profile_set(None, 0)
    e0.record(stream)
    for _ in range(args.steps):
        step(G)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    n_gemm, n_all = ctypes.c_int(0), ctypes.c_int(0)
    lib.gns_profile_query(ctypes.byref(n_gemm), ctypes.byref(n_all))
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    value = whole_job_rate(world, COUNT, ms)
    tflops = world * COUNT * alg_flops_per_matrix() / (ms / 1000.0) / 1e12

    # ---- the same step captured once into a CUDA graph: 5 warm-up replays, then 25 replays
    #      each bracketed by events (per-step median and interquartile range) ----
    def graph_timing(reps=25):
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            gns.muon_step(W, G, M, lr=LR, momentum=MU, ns=ns, workspace=ws, status=status, stream=cap)
        torch.cuda.synchronize()
        for _ in range(5):
            graph.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            graph.replay()
            b.record()
        torch.cuda.synchronize()
        t = sorted(a.elapsed_time(b) for a, b in ev)
        q = lambda f: t[min(reps - 1, int(round(f * (reps - 1))))]
        med = q(0.5)
        del graph
        return {"replays": reps, "median_ms": med, "iqr_ms": [q(0.25), q(0.75)],
                "matrices_per_s_at_median": COUNT / (med / 1000.0)}

    graph = graph_timing()

    # ---- instrumented repeat: CUDA events around every GEMM launch (same stream) ----
    per_step = n_gemm.value // max(args.steps, 1)
    cap = per_step * args.steps
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * cap)]
    for e in evs:  # torch creates the CUDA event on first record
        e.record(stream)
    handles = (ctypes.c_void_p * (2 * cap))(*[ctypes.c_void_p(e.cuda_event) for e in evs])
    torch.cuda.synchronize()
    lib.gns_profile_set(handles, cap)
    for _ in range(args.steps):
        step(G)
    torch.cuda.synchronize()
    lib.gns_profile_set(None, 0)
    gemm_ms = sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(cap)) / args.steps
    gemm_launch_ms = gemm_ms / max(per_step, 1)
    flops_per_launch = COUNT * alg_flops_per_matrix() / max(per_step, 1)
    achieved = flops_per_launch / (gemm_launch_ms / 1000.0) / 1e12
    peak_burst, peak_sus, _, peak_src = load_peaks()
    if args.metric_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "ms_per_step": ms, "steps": args.steps,
                              "warmup": args.warmup, "graph_replay": graph,
                              "gemm_ms_per_step": gemm_ms, "gemm_launches_per_step": per_step,
                              "gemm_frac_of_burst": achieved / peak_burst, "step_frac_of_burst": tflops / peak_burst,
                              "gpu_launches": n_all.value, "clocks": clk, "device_status": int(status.item()),
                              "note": "--metric-only: the metric step alone (for profiling), not a bench line"}),
                  flush=True)
        return 0

    # ---- end to end: gradient in from pinned host memory, weights back, every step ----
    # The copies of step t overlap compute as a training loop would overlap them: the next
    # step's gradient is copied in (double-buffered) while this step runs, and the updated
    # weights are copied out from a device snapshot (double-buffered, so the step after
    # next never waits for this copy) while the next steps run. Every step
    # still moves its whole gradient in and its whole weight matrix out inside the timed
    # region, which ends when the last copy out has finished.
    G_host = G.cpu().pin_memory()
    W_host = torch.empty_like(W, device="cpu").pin_memory()
    G_dev = [torch.empty_like(G), torch.empty_like(G)]
    W_snap = [torch.empty_like(W), torch.empty_like(W)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    barrier()
    ev = lambda: torch.cuda.Event()

    def run_e2e(nsteps):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        in_ready = [ev(), ev()]
        used = [ev(), ev()]        # step that read G_dev[i] is done
        out_done = [ev(), ev()]    # the last copy out of W_snap[i] is done
        with torch.cuda.stream(s_in):
            G_dev[0].copy_(G_host, non_blocking=True)
            in_ready[0].record(s_in)
        out_done[0].record(s_out)
        out_done[1].record(s_out)
        for t in range(nsteps):
            cur, nxt = t % 2, (t + 1) % 2
            if t + 1 < nsteps:
                with torch.cuda.stream(s_in):
                    if t >= 1:
                        s_in.wait_event(used[nxt])
                    G_dev[nxt].copy_(G_host, non_blocking=True)
                    in_ready[nxt].record(s_in)
            stream.wait_event(in_ready[cur])
            step(G_dev[cur])
            used[cur].record(stream)
            stream.wait_event(out_done[cur])
            W_snap[cur].copy_(W, non_blocking=True)
            snap = ev()
            snap.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(snap)
                W_host.copy_(W_snap[cur], non_blocking=True)
                out_done[cur] = ev()
                out_done[cur].record(s_out)
        stream.wait_event(out_done[0])
        stream.wait_event(out_done[1])
        f1.record(stream)
        torch.cuda.synchronize()
        return f0.elapsed_time(f1)

    e2e_steps = max(3, min(args.steps, 20))
    run_e2e(3)  # untimed: first use of the pinned buffers and the copy streams
    barrier()
    e2e_total = run_e2e(e2e_steps)
    barrier()
    e2e_ms = max_over_ranks(e2e_total / e2e_steps)
    bytes_step = COUNT * ROWS * COLS * 2
    del G_dev, W_snap

    # ---- Gram NS against standard NS on the same kernels (orthogonalization only) ----
    X = M.clone()
    out = torch.empty_like(X)
    ws_g = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_GRAM_NS, X, ns), dev)
    ws_s = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_NS_STANDARD, X, ns), dev)

    def time_ns(fn, ws_):
        for _ in range(3):
            fn(X, outs=[out], ns=ns, workspace=ws_, stream=stream)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(10, args.steps // 4)
        a.record(stream)
        for _ in range(reps):
            fn(X, outs=[out], ns=ns, workspace=ws_, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    gram_ms = time_ns(gns.gram_ns_batched, ws_g)
    std_ms = time_ns(gns.ns_standard_batched, ws_s)
    del ws_g, ws_s, X, out

    # ---- the other update flavours on the same workload (whole steps, inputs in HBM) ----
    V = torch.zeros((COUNT, 1, ROWS), dtype=torch.float32, device=dev)

    def time_flavor(params, with_v=False):
        need = gns.workspace_size(_lib.GNS_OP_MUON_STEP, M, ns, muon=params)
        ws_f = gns.alloc_workspace(need, dev)

        def go():
            gns.muon_step(W, G, M, ns=ns, workspace=ws_f, status=status, stream=stream, params=params,
                          V=V if with_v else None)
        for _ in range(3):
            go()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(10, args.steps // 4)
        a.record(stream)
        for _ in range(reps):
            go()
        b.record(stream)
        torch.cuda.synchronize()
        step_ms = a.elapsed_time(b) / reps
        # instrumented repeat: CUDA events around the GEMM launches of each step
        cap = 8 * reps
        evf = [torch.cuda.Event(enable_timing=True) for _ in range(2 * cap)]
        for e in evf:
            e.record(stream)
        hf = (ctypes.c_void_p * (2 * cap))(*[ctypes.c_void_p(e.cuda_event) for e in evf])
        torch.cuda.synchronize()
        lib.gns_profile_set(hf, cap)
        for _ in range(reps):
            go()
        torch.cuda.synchronize()
        ng = ctypes.c_int(0)
        lib.gns_profile_query(ctypes.byref(ng), None)
        lib.gns_profile_set(None, 0)
        n_rec = min(ng.value, cap)
        g_ms = sum(evf[2 * i].elapsed_time(evf[2 * i + 1]) for i in range(n_rec)) / reps
        return step_ms, g_ms

    # ---- the MoE-expert alpha = 4 batch: Gram NS alone on 256 x 2048 x 8192 ----
    def moe_experts():
        count, n, m = 256, 2048, 8192
        X = (torch.randn((count, n, m), generator=gen, device=dev, dtype=torch.float32) / m ** 0.5).to(torch.bfloat16)
        r = {"what": "Gram NS alone (T=5, restart@2) on 256 expert matrices 2048 x 8192 bf16 (alpha = 4), "
                     "N(0,1)/sqrt(m) entries"}
        r.update(time_orth(X, gns.gram_ns_batched, _lib.GNS_OP_GRAM_NS, count * alg_flops_per_matrix(n, m)))
        std = time_orth(X, gns.ns_standard_batched, _lib.GNS_OP_NS_STANDARD, count * std_flops_per_matrix(n, m))
        r["standard_ns_ms_per_call"] = std["ms_per_call"]
        r["gram_vs_standard_speedup"] = std["ms_per_call"] / r["ms_per_call"]
        del X
        torch.cuda.empty_cache()
        return r

    def moe_squares():
        count, n = 64, 7168
        X = (torch.randn((count, n, n), generator=gen, device=dev, dtype=torch.float32) / n ** 0.5).to(torch.bfloat16)
        r = {"what": "standard NS (T=5, symmetric products; alpha = 1, where Gram NS saves nothing) on 64 square "
                     "matrices 7168 x 7168 bf16, N(0,1)/sqrt(n) entries"}
        r.update(time_orth(X, gns.ns_standard_batched, _lib.GNS_OP_NS_STANDARD, count * std_flops_per_matrix(n, n)))
        del X
        torch.cuda.empty_cache()
        return r

    moe = moe_experts()
    moe_sq = moe_squares()

    # ---- many small matrices (one call per batch; products of at most 128 rows take the
    #      1-CTA 128 x 128 tile plan) and a batch-size sweep at 1024 x 4096 ----
    def batch_sweep():
        res = {}
        n, m = ROWS, COLS
        for count in [1, 2, 4, 8, 16, 24, 32, 48, 64]:
            X = (torch.randn((count, n, m), generator=gen, device=dev, dtype=torch.float32) / m ** 0.5).to(
                torch.bfloat16)
            r = time_orth(X, gns.gram_ns_batched, _lib.GNS_OP_GRAM_NS, count * alg_flops_per_matrix(n, m))
            res[str(count)] = {k: r[k] for k in ("ms_per_call", "matrices_per_s", "gemm_tflops",
                                                 "gemm_frac_of_burst_peak")}
            del X
            torch.cuda.empty_cache()
        return res

    small = small_batches()
    sweep = batch_sweep()

    # ---- the fractional-update configuration: 32 x 4096 x 16384, f = 1/4 (k = 1024) ----
    def frac_config(rows=4096, cols=16384):
        count = 32
        sc = 1.0 / cols ** 0.5

        def rnd():
            return (torch.randn((count, rows, cols), generator=gen, device=dev, dtype=torch.float32) * sc).to(
                torch.bfloat16)
        Wf, Gf, Mf = rnd(), rnd(), rnd()
        pf = gns.MuonParams(lr=LR, momentum=MU, frac=0.25)
        ws_f = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_MUON_STEP, Mf, ns, muon=pf), dev)

        def go():
            gns.muon_step(Wf, Gf, Mf, ns=ns, workspace=ws_f, status=status, stream=stream, params=pf)
        for _ in range(2):
            go()
        torch.cuda.synchronize()
        reps = 5
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            go()
        b.record(stream)
        torch.cuda.synchronize()
        f_ms = a.elapsed_time(b) / reps
        n, m = min(rows, cols), max(rows, cols)
        k = (n + 3) // 4
        fl = count * alg_flops_per_matrix(k, m)
        del Wf, Gf, Mf, ws_f
        torch.cuda.empty_cache()
        sel = "rows" if rows <= cols else "columns (the rows of the transpose)"
        return {"what": f"Dion3 fractional update f = 1/4 on 32 bf16 momentum matrices {rows} x {cols}: exact l1 "
                        f"top-{k} {sel}, Gram NS of the {k} x {m} subsets, scatter, error feedback",
                "ms_per_step": f_ms, "matrices_per_s": count / (f_ms / 1000.0),
                "orthogonalization_tflops_over_step": fl / (f_ms / 1000.0) / 1e12}

    frac_cfg = frac_config()
    frac_tall = frac_config(16384, 4096)

    # ---- the mixed dense-transformer layer set: 32 layers of one 4096 x 4096 (alpha = 1,
    # standard NS) and two 4096 x 11008 plus one 11008 x 4096 (alpha = 2.69, Gram NS) ----
    def dense_layers():
        shapes = [(32, 4096, 4096), (64, 4096, 11008), (32, 11008, 4096)]

        def rnd(sh):
            return (torch.randn(sh, generator=gen, device=dev, dtype=torch.float32) / sh[2] ** 0.5).to(torch.bfloat16)
        Ws = [rnd(sh) for sh in shapes]
        Gs = [rnd(sh) for sh in shapes]
        Ms = [rnd(sh) for sh in shapes]
        pd = gns.MuonParams(lr=LR, momentum=MU)
        ws_d = gns.alloc_workspace(gns.workspace_size(_lib.GNS_OP_MUON_STEP, Ms, ns, muon=pd), dev)

        def go():
            gns.muon_step(Ws, Gs, Ms, ns=ns, workspace=ws_d, status=status, stream=stream, params=pd)
        go()
        torch.cuda.synchronize()
        reps = 3
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            go()
        b.record(stream)
        torch.cuda.synchronize()
        d_ms = a.elapsed_time(b) / reps
        fl = 0.0
        for (c, r, k) in shapes:
            n, m = min(r, k), max(r, k)
            fl += c * ((5 * (3 * m / n + 1)) * n ** 3 if n == m else alg_flops_per_matrix(n, m))
        del Ws, Gs, Ms, ws_d
        torch.cuda.empty_cache()
        return {"what": "one Muon step over 32 layers x {4096 x 4096, 2 x 4096 x 11008, 11008 x 4096} bf16 "
                        "(squares by standard NS with symmetric products, the rest by Gram NS)",
                "ms_per_step": d_ms, "matrices_per_s": 128 / (d_ms / 1000.0),
                "algorithmic_tflops_over_step": fl / (d_ms / 1000.0) / 1e12}

    dense = dense_layers()

    base = dict(lr=LR, momentum=MU)
    f16_ms, f16_gemm = time_flavor(gns.MuonParams(**base, ns_dtype=torch.float16))
    normuon_ms, normuon_gemm = time_flavor(gns.MuonParams(**base, flavor="normuon", beta2=0.95, norm_eps=1e-8),
                                           with_v=True)
    rownorm_ms, _ = time_flavor(gns.MuonParams(**base, flavor="rownorm", rownorm_gamma=0.15, norm_eps=1e-8))
    frac_ms, _ = time_flavor(gns.MuonParams(**base, frac=0.25))
    step_flops = COUNT * alg_flops_per_matrix()

    # Periodic Row-wise Muon, K = 3: the three steps of one period (Newton-Schulz on t = 0,
    # RowNorm on t = 1, 2), each timed, over several periods
    def periodic_timing(periods=10):
        pp = [gns.MuonParams(**base, flavor="periodic", period=3, step=t, rownorm_gamma=0.15, norm_eps=1e-8)
              for t in range(3)]
        ws_p = gns.alloc_workspace(max(gns.workspace_size(_lib.GNS_OP_MUON_STEP, M, ns, muon=p) for p in pp), dev)
        for p in pp:
            gns.muon_step(W, G, M, ns=ns, workspace=ws_p, status=status, stream=stream, params=p)
        torch.cuda.synchronize()
        evp = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
               for _ in range(periods)]
        for per in evp:
            for t, (a, b) in enumerate(per):
                a.record(stream)
                gns.muon_step(W, G, M, ns=ns, workspace=ws_p, status=status, stream=stream, params=pp[t])
                b.record(stream)
        torch.cuda.synchronize()
        per_t = [sum(per[t][0].elapsed_time(per[t][1]) for per in evp) / periods for t in range(3)]
        return {"ms_per_step_t0_ns": per_t[0], "ms_per_step_t1_rownorm": per_t[1], "ms_per_step_t2_rownorm": per_t[2],
                "mean_ms_per_step": sum(per_t) / 3.0, "periods_timed": periods,
                "what": "Periodic Row-wise Muon (K = 3, gamma = 0.15): each step of a period timed with CUDA events"}

    periodic = periodic_timing()

    def gemm_roofline(g_ms, what):
        ach = step_flops / (g_ms / 1000.0) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": peak_burst, "unit": "TFLOP/s", "frac": ach / peak_burst,
                "frac_of_sustained": ach / peak_sus, "gemm_ms_per_step": g_ms, "kernel": what,
                "peak_kind": f"dense bf16 burst, {peak_src} (fp16 dense rate = bf16 dense rate)"}
    _, _, hbm_peak, _ = load_peaks()
    # RowNorm step: algorithmic traffic = read G, M, W and write M, W once (bf16)
    rn_bytes = COUNT * ROWS * COLS * 2 * 5
    flavors = {
        "note": "whole optimizer steps on the same 24 x 1024 x 4096 bf16 workload, inputs in HBM",
        "fp16_products": {"ms_per_step": f16_ms, "matrices_per_s": COUNT / (f16_ms / 1000.0),
                          "what": "Muon step with the Newton-Schulz products in fp16 (the float16 cast of Dion3 Algorithm 3)",
                          "roofline": gemm_roofline(f16_gemm, "gns::tc::gemm_kernel, fp16 operands")},
        "normuon": {"ms_per_step": normuon_ms, "matrices_per_s": COUNT / (normuon_ms / 1000.0),
                    "what": "NorMuon (Dion3 eq. (2)): Gram NS to O, row second moments, row scaling, update",
                    "roofline": gemm_roofline(normuon_gemm, "gns::tc::gemm_kernel, bf16, O written for the "
                                                            "NorMuon statistics")},
        "rownorm": {"ms_per_step": rownorm_ms, "matrices_per_s": COUNT / (rownorm_ms / 1000.0),
                    "what": "RowNorm off-refresh step (Scaling Muon for DiTs eq. (5), (7))",
                    "roofline": {"bound": "hbm", "achieved": rn_bytes / (rownorm_ms / 1000.0) / 1e9,
                                 "peak": hbm_peak, "unit": "GB/s",
                                 "frac": rn_bytes / (rownorm_ms / 1000.0) / 1e9 / hbm_peak,
                                 "algorithmic_bytes": rn_bytes}},
        "periodic_K3": periodic,
        "frac_quarter": {"ms_per_step": frac_ms, "matrices_per_s": COUNT / (frac_ms / 1000.0),
                         "what": "Dion3 fractional update, f = 1/4 (Algorithm 4, Muon flavour)"},
    }
    del V

    st = int(status.item())
    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        # whole 24-matrix steps of the oracle until at least 10 s of CPU work
        n_cpu, t = 0, 0.0
        while t < 10.0 and n_cpu < 20 * COUNT:
            t += time_oracle(COUNT, seed=1 + n_cpu)
            n_cpu += COUNT
        cpu = {"value": n_cpu / t, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n_cpu // COUNT} full 24-matrix Muon steps in the fp64 numpy oracle "
                         f"({t:.1f} s)"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world),
        "tflops": tflops, "tflops_frac_of_peak": tflops / peak_burst,
        "e2e": {"value": whole_job_rate(world, COUNT, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": bytes_step,
                "d2h_bytes_per_step": bytes_step, "ms_per_step": e2e_ms,
                "how": "gradient H2D from pinned host memory (double-buffered, overlapping the previous step) and "
                       "updated weights D2H from double-buffered device snapshots (overlapping the next steps), "
                       "every step"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": achieved / peak_burst, "traffic": gemm_traffic() if per_step == 1 else None,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, captured on "
                                       f"this kernel code ({gemm_source_hash()}: the sources' sha256 prefix with "
                                       "comments removed) by bench.py --metric-only; null when no capture of this "
                                       "code is on record",
                     "kernel": f"gns::tc::gemm_kernel (tcgen05 bf16 GEMM; {per_step} launch(es) per step carry the 17 products)",
                     "peak_kind": f"dense bf16 burst, {peak_src}",
                     "frac_of_sustained": achieved / peak_sus,
                     "gemm_ms_per_step": gemm_ms, "gemm_launches_per_step": per_step},
        "graph_replay": graph,
        "gram_vs_standard": {"gram_ns_ms": gram_ms, "standard_ns_ms": std_ms, "speedup": std_ms / gram_ms,
                             "note": "orthogonalization of the 24 matrices alone, same tcgen05 kernels, T=5; "
                                     "standard NS with symmetric products (Dion3 Algorithm 1, sec. 2.3)"},
        "flavors": flavors,
        "moe_experts_alpha4": moe,
        "moe_squares_7168": moe_sq,
        "small_matrices": small,
        "batch_sweep_1024x4096_gram_ns": sweep,
        "frac_quarter_4096x16384": frac_cfg,
        "frac_quarter_16384x4096_tall": frac_tall,
        "dense_layers_32": dense,
        "gpu_launches": n_all.value,
        "device_status": st,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--metric-only", action="store_true",
                    help="time the metric step alone and print a short line (for profiling runs)")
    ap.add_argument("--small-only", action="store_true",
                    help="time the small-matrix section alone and print it (for profiling runs)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group(backend=backend)
        dist = tdist
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
