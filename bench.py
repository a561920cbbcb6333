#!/usr/bin/env python3
"""Decode-step benchmark for libpnq on GB300.

Workload: a Qwen-27B-shaped decode step, 64 layers x 7 projections, every projection a
separate pnq_gemv call (pn3t gate/up [17408x5120], q [12288x5120]; pn4t k/v [1024x5120],
o [5120x6144], down [5120x17408]); 11.0 GB of weights generated on the device from a seed
(codes uniform, d = fp16(+-|N(0, 0.003)|), pn3t reserved bits clear); x ~ N(0, 1) fp32;
M = 1 by default. One step = all 448 GEMVs, captured once in a CUDA graph and replayed.
The weights are 85x the L2, so every replay reads them from HBM (no flush needed).

Reported (one JSON line from rank 0): weight GB/s over the step (value), us per step,
fraction of the measured HBM copy bandwidth, an end-to-end figure through the C ABI with
the step's activations copied from pinned host memory and the last output copied back,
the dominant kernel's roofline measured with CUDA events, SM clocks sampled during the
timed region, and the CPU oracle on a bounded sample of the same workload.

--impl reference times the CPU oracle (oracle/) on the same workload, one sampled layer
per step. With N > 1 (torchrun), every rank runs an independent replica of the step
(the GEMV has no exchange step) and value is the bytes of all ranks over the slowest rank.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

PN3T, PN4T, NVFP4 = 124, 125, 1004
BLK = {PN3T: 80, PN4T: 64}
# name, type, N, K
PROJECTIONS = [("attn_q", PN3T, 12288, 5120), ("attn_k", PN4T, 1024, 5120), ("attn_v", PN4T, 1024, 5120),
               ("attn_o", PN4T, 5120, 6144), ("ffn_gate", PN3T, 17408, 5120), ("ffn_up", PN3T, 17408, 5120),
               ("ffn_down", PN4T, 5120, 17408)]
METRIC = "GEMV weight GB/s and % of GB300 HBM peak at M=1; us per 27B-shaped decode step"
SEED = 20261202
L2_BYTES = 129e6  # GB300 L2 size in bytes


def row_bytes(t, K):
    return K // BLK[t] * 34


def layer_bytes():
    return sum(N * row_bytes(t, K) for _, t, N, K in PROJECTIONS)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------- helpers

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="pnq_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
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
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def kernel_source_digest():
    h = hashlib.sha256()
    for fn in ("pnq_gemv_pn.cu", "pnq_cluster.cuh", "pnq_split.cuh", "pnq_device.cuh"):
        with open(os.path.join(ROOT, "block_quantized_weight_pn3t_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str):
    """dram bytes per launch for the dominant kernel from the committed ncu summary, or None when
    the summary is missing or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"kernel_source_digest:\s*`?([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*`?([0-9.e+]+)", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_digest():
        return None
    return float(m_tr.group(1))


def workload_config(M: int, L: int, n_calls: int, world: int) -> dict:
    """The `config` object both arms report: the decode-step workload and how it is run."""
    step_bytes = L * layer_bytes()
    return {"workload": "qwen27b-decode-step-64x7", "layers": L, "M": M,
            "projections": {n: f"{'pn3t' if t == PN3T else 'pn4t'} {N}x{K}" for n, t, N, K in PROJECTIONS},
            "weight_bytes_per_step": step_bytes,
            "l2": f"inputs larger than L2 (weights {step_bytes / L2_BYTES:.1f}x the L2 per step); no flush",
            "graph": f"one CUDA graph per step, {n_calls} pnq_gemv launches", "parallelism": f"replicas x{world}"}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------- CPU oracle legs

def host_layer(layer: int):
    """One layer's weights regenerated on the host (identical bytes to the device replica)."""
    from block_quantized_weight_pn3t_gb300 import synth
    out = []
    for p, (name, t, N, K) in enumerate(PROJECTIONS):
        out.append(synth.pn_random_blocks(t, N, K, seed=SEED, stream=layer * 8 + p).numpy())
    return out


def host_x(M):
    from block_quantized_weight_pn3t_gb300 import synth
    return {K: synth.activations(M, K, seed=SEED + K) for K in sorted({K for *_, K in PROJECTIONS})}


def oracle_layer(oracle, layer_w, xs):
    nbytes = 0
    for (name, t, N, K), W in zip(PROJECTIONS, layer_w):
        oracle.gemv(t, W, N, K, xs[K])
        nbytes += W.nbytes
    return nbytes


def cpu_baseline(M: int, budget_s: float = 12.0):
    """The oracle (single-threaded C, fp64) on whole sampled layers until ~budget_s of CPU time on one
    core, then the same oracle on every host core (one spawned process per core, rows split evenly,
    a barrier before the timed part): the all-cores figure is the line's value."""
    import oracle
    oracle.lib()
    xs = host_x(M)
    nbytes, elapsed, layers = 0, 0.0, 0
    while elapsed < budget_s and layers < 64:
        w = host_layer(layers)
        t0 = time.perf_counter()
        nbytes += oracle_layer(oracle, w, xs)
        elapsed += time.perf_counter() - t0
        layers += 1
    one = {"value": round(nbytes / elapsed / 1e9, 5), "unit": "GB/s", "cores": 1,
           "sample": f"layers 0..{layers - 1} of 64 (all 7 projections, {nbytes / 1e6:.0f} MB of weights), M={M}, "
                     f"{elapsed:.1f} s of single-thread fp64 CPU work"}
    try:
        allc = cpu_baseline_all_cores(M)
    except Exception as e:  # the single-core figure stands alone
        return dict(one, kind="oracle", all_cores_error=str(e)[:200])
    return dict(allc, kind="oracle", single_core=one)


def _oracle_worker_init(barrier):
    global _BARRIER
    _BARRIER = barrier


def _oracle_worker(task):
    """One host core: regenerate its rows of the sampled layers, wait for the others, then run the
    oracle on them; returns (weight bytes, seconds of oracle work)."""
    import oracle
    from block_quantized_weight_pn3t_gb300 import synth
    M, layers, worker, workers = task
    oracle.lib()
    xs = host_x(M)
    work = []
    for layer in range(layers):
        for p, (name, t, N, K) in enumerate(PROJECTIONS):
            r0, r1 = N * worker // workers, N * (worker + 1) // workers
            if r1 > r0:
                rows = torch.arange(r0, r1, dtype=torch.int64)
                work.append((t, synth.pn_random_blocks(t, N, K, seed=SEED, stream=layer * 8 + p, rows=rows).numpy(),
                             r1 - r0, K))
    _BARRIER.wait()
    t0 = time.perf_counter()
    nbytes = 0
    for t, W, n, K in work:
        oracle.gemv(t, W, n, K, xs[K])
        nbytes += W.nbytes
    return nbytes, time.perf_counter() - t0


def cpu_baseline_all_cores(M: int, layers: int = 8):
    import concurrent.futures
    import multiprocessing
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    ctx = multiprocessing.get_context("spawn")
    barrier = ctx.Barrier(cores)
    with concurrent.futures.ProcessPoolExecutor(cores, mp_context=ctx, initializer=_oracle_worker_init,
                                                initargs=(barrier,)) as ex:
        res = list(ex.map(_oracle_worker, [(M, layers, w, cores) for w in range(cores)]))
    nbytes = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    return {"value": round(nbytes / wall / 1e9, 5), "unit": "GB/s", "cores": cores,
            "sample": f"layers 0..{layers - 1} of 64 (all 7 projections, {nbytes / 1e6:.0f} MB of weights), M={M}, "
                      f"rows split over {cores} spawned processes (one per core), {wall:.2f} s wall "
                      f"(slowest process) of fp64 CPU work"}


REF_ROW_FRACTION = 16  # the reference arm's step: the first 1/16 of every projection's rows of layer 0


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from block_quantized_weight_pn3t_gb300 import synth
    oracle.lib()
    xs = host_x(args.m)
    sample = []
    for p, (name, t, N, K) in enumerate(PROJECTIONS):
        n = max(1, N // REF_ROW_FRACTION)
        W = synth.pn_random_blocks(t, N, K, seed=SEED, stream=p, rows=torch.arange(n, dtype=torch.int64)).numpy()
        sample.append((t, W, n, K))

    def step():
        nb = 0
        for t, W, n, K in sample:
            oracle.gemv(t, W, n, K, xs[K])
            nb += W.nbytes
        return nb

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += step()
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample_bytes = sum(W.nbytes for _, W, _, _ in sample)
    desc = (f"the first 1/{REF_ROW_FRACTION} of the rows of each of layer 0's 7 projections "
            f"({sample_bytes / 1e6:.1f} MB of weights) per step, M={args.m}, one host core")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(args.m, args.layers, args.layers * len(PROJECTIONS), args.gpus),
                           sample=desc),
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{desc}, {args.steps} steps"},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------- GPU arm

def aggregate_replicas(times_ms, world, step_bytes, pg=None, device=None):
    """Whole-job figures of `world` replicas of the step: each time is the slowest rank's (max over
    ranks; pg = torch.distributed or None), each throughput = the bytes of all replicas / it."""
    t = torch.tensor([float(v) for v in times_ms], dtype=torch.float64, device=device)
    if pg is not None:
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
    slowest = [float(v) for v in t.cpu()]
    return slowest, [world * step_bytes / (v * 1e-3) / 1e9 for v in slowest]


def graph_us_per_launch(launch, n_launch, stream, reps, warmup):
    """launch(h) issues n_launch GEMVs on stream handle h; captured once in a CUDA graph, replayed
    `warmup` times, then `reps` replays timed with CUDA events on the replay stream: us per GEMV."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        launch(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * n_launch)


SINGLE_SHAPES = [("pn4t 5120x17408 M=1 (down-projection shape)", PN4T, 5120, 17408),
                 ("nvfp4 17408x5120 M=1", NVFP4, 17408, 5120), ("nvfp4 5120x17408 M=1", NVFP4, 5120, 17408)]


def single_call_lines(dev, stream, flags, peak, warmup, M=1):
    """One GEMV shape at a time (M activation rows, the same flags as the step), called back to
    back in a graph that rotates through weight copies whose total exceeds the L2 twice (so every
    call reads HBM): us per call, weight GB/s and the fraction of the measured HBM rate."""
    import block_quantized_weight_pn3t_gb300 as pnq
    from block_quantized_weight_pn3t_gb300 import synth
    out = []
    for label, t, N, K in SINGLE_SHAPES:
        wbytes = N * K // 2 + N * K // 16 if t == NVFP4 else N * row_bytes(t, K)
        n_copies = max(3, -(-int(2 * L2_BYTES) // wbytes))
        if t == NVFP4:
            ws = [synth.nvfp4_random(N, K, seed=SEED, stream=c, device=dev) for c in range(n_copies)]
            descs = [pnq.nvfp4_weights(c.data_ptr(), sc.data_ptr(), g) for c, sc, g in ws]
            X = torch.from_numpy(synth.activations_bf16(M, K, seed=SEED).view(np.int16)).to(dev)
        else:
            ws = [synth.pn_random_blocks(t, N, K, seed=SEED, stream=c, device=dev) for c in range(n_copies)]
            descs = [w.data_ptr() for w in ws]
            X = torch.from_numpy(synth.activations(M, K, seed=SEED)).to(dev)
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        n = n_copies * max(1, 60 // n_copies)

        def launch(h):
            for i in range(n):
                rc = pnq.gemv_ex_ptr(t, descs[i % n_copies], N, K, X.data_ptr(), M, Y.data_ptr(), flags, h)
                if rc != 0:
                    raise pnq.PnqError("pnq_gemv", rc)

        us = graph_us_per_launch(launch, n, stream, reps=5, warmup=warmup)
        gbs = wbytes / (us * 1e-6) / 1e9
        out.append({"shape": label.replace("M=1", f"M={M}"), "us_per_call": round(us, 3), "weight_bytes": wbytes, "achieved": round(gbs, 1),
                    "frac": round(gbs / peak, 4), "weight_copies": n_copies, "launches": n})
        del ws
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import block_quantized_weight_pn3t_gb300 as pnq
    from block_quantized_weight_pn3t_gb300 import synth

    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the libpnq arm")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    pnq.lib()
    M, L = args.m, args.layers

    # ---- inputs resident in HBM: weights, activations, outputs
    weights = []  # [layer][proj] -> uint8 tensor
    for layer in range(L):
        weights.append([synth.pn_random_blocks(t, N, K, seed=SEED, stream=layer * 8 + p, device=dev)
                        for p, (_, t, N, K) in enumerate(PROJECTIONS)])
    step_bytes = L * layer_bytes()
    xs_host = host_x(M)
    xs = {K: torch.from_numpy(v).to(dev) for K, v in xs_host.items()}
    ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for (_, _, N, _) in PROJECTIONS]
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    calls = []
    for layer in range(L):
        for p, (_, t, N, K) in enumerate(PROJECTIONS):
            calls.append((t, weights[layer][p].data_ptr(), N, K, xs[K].data_ptr(), ys[p].data_ptr()))

    # model weights do not change inside the decode loop: let each GEMV stream its weights while
    # the previous one finishes (x is still read only after it completes)
    flags = pnq.GEMV_STATIC_WEIGHTS

    def issue(seq, h):
        """The GEMVs of seq, in order, on stream handle h."""
        for t, w, N, K, x, y in seq:
            rc = pnq.gemv_ex_ptr(t, w, N, K, x, M, y, flags, h)
            if rc != 0:
                raise pnq.PnqError("pnq_gemv", rc)

    def step(s):
        issue(calls, s.cuda_stream)

    # eager warm-up (sets kernel attributes once), then capture one step in a graph
    with torch.cuda.stream(stream):
        step(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays, events on the replay stream
    sampler = ClockSampler(local)
    sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    clocks = sampler.stop()

    # ---- end to end through the C ABI: activations from pinned host memory, last output back
    xs_pinned = {K: torch.from_numpy(v).pin_memory() for K, v in xs_host.items()}
    y_last = torch.empty((M, PROJECTIONS[-1][2]), dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * 4 for v in xs_pinned.values())
    d2h = y_last.numel() * 4
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_step():
        for K, v in xs_pinned.items():
            xs[K].copy_(v, non_blocking=True)
        graph.replay()
        y_last.copy_(ys[-1], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        stream.synchronize()
        if pg:
            pg.barrier()
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps

    # ---- dominant kernel (the pn3t GEMV): the step's 192 pn3t launches in their stream order and
    # with the same flags, captured back to back in a graph of their own; events on the replay
    # stream around the replays give the average launch duration
    dom = [(t, w, N, K, x, y) for (t, w, N, K, x, y) in calls if t == PN3T]

    def dom_launches(h):
        issue(dom, h)

    gdom = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gdom, stream=stream):
        dom_launches(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        gdom.replay()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        d0.record(stream)
        for _ in range(args.steps):
            gdom.replay()
        d1.record(stream)
    torch.cuda.synchronize()
    dur_ms = [d0.elapsed_time(d1) / (args.steps * len(dom))] * len(dom)
    dom_bytes = sum(N * row_bytes(t, K) for (t, _, N, K, _, _) in dom)
    dom_gbs = dom_bytes / (sum(dur_ms) * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    traffic = profiled_traffic("pn3t_gemv_m1_decode_step") if M == 1 else None

    # ---- each projection's launches of the step (one per layer) back to back in a graph of their own
    per_proj = {}
    for p, (name, t, N, K) in enumerate(PROJECTIONS):
        sub = calls[p::len(PROJECTIONS)]

        def launch(h, sub=sub):
            issue(sub, h)

        us = graph_us_per_launch(launch, len(sub), stream, reps=max(3, args.steps // 20), warmup=args.warmup)
        gbs = N * row_bytes(t, K) / (us * 1e-6) / 1e9
        per_proj[name] = {"us_per_call": round(us, 3), "achieved": round(gbs, 1), "frac": round(gbs / peak, 4)}
    singles = single_call_lines(dev, stream, flags, peak, args.warmup, M) if not args.no_singles else None

    err = pnq.device_error()
    if err:
        raise SystemExit(f"libpnq recorded a device error (site {err})")

    # ---- aggregate over ranks (replicas): bytes of all ranks / slowest rank
    (ms_max, ms_e2e_max), (value, e2e_value) = aggregate_replicas([ms, ms_e2e], world, step_bytes, pg, dev)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16-mma/f32-acc", "data": "synthetic",
            "config": dict(workload_config(M, L, len(calls), world), us_per_step=round(ms_max * 1e3, 2),
                           hbm_fraction=round(value / world / peak, 4)),
            "roofline": {"bound": "hbm", "achieved": round(dom_gbs, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(dom_gbs / peak, 4), "traffic": traffic,
                         "kernel": (f"pn_rows_kernel<pn3t, NT={1 if M <= 4 else 2}> (row stream, mma.sync decode)"
                                    if M <= 8 else "cluster_gemv_kernel<PnMma<pn3t, NT=4>> (strip pipeline)"),
                         "launches": len(dom),
                         "algorithmic_bytes_per_launch": round(dom_bytes / len(dom)),
                         "avg_launch_us": round(sum(dur_ms) / len(dur_ms) * 1e3, 3),
                         "timing": f"graph of the step's {len(dom)} pn3t launches replayed back to back, "
                                   f"events around {args.steps} replays",
                         "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e_max, 4)},
            "gpu_launches": args.steps * len(calls),
            "clocks": clocks,
            "per_projection": {"timing": f"each projection's {L} launches of the step captured back to back in a "
                                         f"graph of their own (same flags), events around the replays",
                               "unit": "us per call; weight GB/s; fraction of the measured HBM rate", **per_proj},
        }
        if singles is not None:
            line["single_calls"] = singles
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(M)
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


NVFP4_SHAPES = {"nvfp4_17408x5120": (17408, 5120), "nvfp4_5120x17408": (5120, 17408)}


def run_single_nvfp4(args):
    """One NVFP4 GEMV (the NVFP4 workload: codes uniform, e4m3 scales of |N(0,1)|, g = 0.01, bf16
    x), called --warmup times on the default stream: the small case of the NVFP4 ncu summary."""
    import block_quantized_weight_pn3t_gb300 as pnq
    from block_quantized_weight_pn3t_gb300 import synth
    N, K = NVFP4_SHAPES[args.single]
    torch.cuda.set_device(0)
    codes, scales, g = synth.nvfp4_random(N, K, seed=SEED, device="cuda")
    X = torch.from_numpy(synth.activations_bf16(args.m, K, seed=SEED).view(np.int16)).cuda()
    Y = torch.empty((args.m, N), dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        pnq.gemv(pnq.NVFP4, (codes, scales, g), X, N, K, Y=Y, flags=pnq.GEMV_STATIC_WEIGHTS)
    torch.cuda.synchronize()
    err = pnq.device_error()
    print(json.dumps({"single": args.single, "type": pnq.NVFP4, "N": N, "K": K, "M": args.m, "launches": args.warmup,
                      "weight_bytes": codes.numel() + scales.numel(), "device_error": err}))
    if err:
        raise SystemExit(1)


def run_single(args):
    """One projection of layer 0, called a few times on the default stream: the small case the
    committed ncu summaries are captured on (one kernel, few launches, a few GB at most)."""
    import block_quantized_weight_pn3t_gb300 as pnq
    from block_quantized_weight_pn3t_gb300 import synth
    names = [p[0] for p in PROJECTIONS]
    if args.single in NVFP4_SHAPES:
        return run_single_nvfp4(args)
    if args.single not in names:
        raise SystemExit(f"--single must be one of {names + list(NVFP4_SHAPES)}")
    p = names.index(args.single)
    _, t, N, K = PROJECTIONS[p]
    torch.cuda.set_device(0)
    W = synth.pn_random_blocks(t, N, K, seed=SEED, stream=p, device="cuda")
    X = torch.from_numpy(host_x(args.m)[K]).cuda()
    Y = torch.empty((args.m, N), dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        pnq.gemv(t, W, X, N, K, Y=Y, flags=pnq.GEMV_STATIC_WEIGHTS)
    torch.cuda.synchronize()
    err = pnq.device_error()
    print(json.dumps({"single": args.single, "type": t, "N": N, "K": K, "M": args.m, "launches": args.warmup,
                      "weight_bytes": N * row_bytes(t, K), "device_error": err}))
    if err:
        raise SystemExit(1)


PREFILL_SHAPES = [("ffn_gate", PN3T, 17408, 5120), ("ffn_down", PN4T, 5120, 17408)]


def run_prefill(args):
    """The prefill path (pnq_gemm, any M, tcgen05 tf32 splits) on the gate and down shapes at M = 64
    and 512: one JSON line each. Time = mean of CUDA events around one replay of a graph of
    `--steps` back-to-back calls (scratch sized for the whole matrix, allocated once, outside the
    timed region), after `--warmup` calls. useful TFLOP/s counts 2 M N K; the MMAs execute three
    times that (hi x hi, hi x lo, lo x hi), against tf32 tensor throughput = the measured bf16
    peak x the nominal tf32 / bf16 ratio (1.1 / 2.25)."""
    import block_quantized_weight_pn3t_gb300 as pnq
    from block_quantized_weight_pn3t_gb300 import synth
    torch.cuda.set_device(0)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        bf16_kind = "measured"
    except Exception:
        bf16, bf16_kind = 1900.0, "fallback"
    tf32 = bf16 * 1.1 / 2.25
    for name, t, N, K in PREFILL_SHAPES:
        W = synth.pn_random_blocks(t, N, K, seed=SEED, device="cuda")
        for M in (64, 512):
            X = torch.from_numpy(synth.activations(M, K, seed=1)).cuda()
            Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            scratch = torch.empty((pnq.gemm_scratch_bytes(t, N, K, M),), dtype=torch.uint8, device="cuda")
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(args.warmup):
                    pnq.gemm(t, W, X, N, K, Y=Y, scratch=scratch)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(args.steps):
                    pnq.gemm(t, W, X, N, K, Y=Y, scratch=scratch)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            err = pnq.device_error()
            us = e0.elapsed_time(e1) * 1e3 / args.steps
            useful = 2.0 * M * N * K / (us * 1e-6) / 1e12
            print(json.dumps({"op": "prefill_gemm", "projection": name, "type": "pn3t" if t == PN3T else "pn4t",
                              "N": N, "K": K, "M": M, "calls": args.steps, "us_per_call": round(us, 2),
                              "useful_tflops": round(useful, 1), "mma_tflops": round(3 * useful, 1),
                              "bound": "tensor", "peak": round(tf32, 1), "unit": "TFLOP/s",
                              "frac": round(3 * useful / tf32, 4),
                              "peak_source": f"MEASURED_PEAKS.json bf16_tflops x 1.1/2.25 ({bf16_kind})",
                              "includes": "x split, slice decode to two tf32 planes, GEMM", "device_error": err}),
                  flush=True)
            del g, scratch
        del W
        torch.cuda.empty_cache()


CODEC_SHAPES = [(PN4T, 5120, 17408), (PN3T, 17408, 5120), (NVFP4, 17408, 5120)]


def run_codec(args):
    """Dequantize and validate on full-size shapes (pn4t 5120 x 17408, pn3t 17408 x 5120, NVFP4
    17408 x 5120; weights generated on the device from the seed). Each call's time is the mean of
    CUDA events around one replay of a CUDA graph of back-to-back calls (`--steps`, at least one
    per weight copy; captured after `--warmup` calls), rotating through weight copies that
    together exceed the L2 twice, so the weights come from HBM.
    Algorithmic bytes per call: the weights read plus the fp32 weights written (dequantize); for
    validate, the int32 row flags written plus the PN tensor (its d fields sit at a 34-byte stride,
    so every 32-byte sector holds one and the whole tensor crosses the bus) or the NVFP4 scales
    alone. One JSON line per operation and shape."""
    import block_quantized_weight_pn3t_gb300 as pnq
    from block_quantized_weight_pn3t_gb300 import synth
    torch.cuda.set_device(0)
    peak, peak_kind = measured_peaks()
    out = None
    for t, N, K in CODEC_SHAPES:
        if t == NVFP4:
            wbytes = N * K // 2 + N * K // 16
            name = "nvfp4"
        else:
            wbytes = N * row_bytes(t, K)
            name = "pn3t" if t == PN3T else "pn4t"
        n_copies = max(2, -(-int(2 * L2_BYTES) // wbytes))
        if t == NVFP4:
            # validate reads only the scales: enough distinct scale tensors for them alone to
            # exceed the L2 twice, paired with the code tensors in rotation
            n_codes = n_copies
            n_copies = max(n_codes, -(-int(2 * L2_BYTES) // (N * K // 16)))
            gen = [synth.nvfp4_random(N, K, seed=SEED, stream=c, device="cuda") for c in range(n_codes)]
            more = [synth.nvfp4_random(N, K, seed=SEED, stream=c, device="cuda")[1] for c in range(n_codes, n_copies)]
            copies = [(gen[c % n_codes][0], gen[c][1] if c < n_codes else more[c - n_codes], gen[0][2])
                      for c in range(n_copies)]
        else:
            copies = [synth.pn_random_blocks(t, N, K, seed=SEED, stream=c, device="cuda") for c in range(n_copies)]
        if out is None or out.numel() < N * K:
            out = torch.empty((N * K,), dtype=torch.float32, device="cuda")
        flags = torch.empty((N,), dtype=torch.int32, device="cuda")
        ops = [("dequantize_row", lambda W: pnq.dequantize_row(t, W, N, K, out=out[:N * K].view(N, K)),
                wbytes + 4 * N * K),
               ("validate_row", lambda W: pnq.validate_row(t, W, N, K, flags=flags),
                (N * K // 16 if t == NVFP4 else wbytes) + 4 * N)]
        for op, call, nbytes in ops:
            reps = max(args.steps, n_copies)  # every copy at least once, none reused while in L2
            # the calls are captured once into a CUDA graph and replayed, so the time is the
            # device's (a Python call costs more than a small kernel)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for i in range(args.warmup):
                    call(copies[i % n_copies])
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(args.warmup, args.warmup + reps):
                    call(copies[i % n_copies])
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / reps
            del g
            gbs = nbytes / (us * 1e-6) / 1e9
            print(json.dumps({"op": op, "type": name, "N": N, "K": K, "calls": reps, "us_per_call": round(us, 3),
                              "algorithmic_bytes": nbytes, "weight_copies": n_copies, "achieved": round(gbs, 1),
                              "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                              "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"}), flush=True)
        del copies
        torch.cuda.empty_cache()
    err = pnq.device_error()
    if err:
        raise SystemExit(f"libpnq recorded a device error (site {err})")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--m", type=int, default=1, help="activation rows (1..16)")
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-singles", action="store_true", help="skip the single-GEMV lines of the JSON line")
    ap.add_argument("--prefill", action="store_true",
                    help="time the prefill path (pnq_gemm) on the gate and down shapes at M = 64 and 512")
    ap.add_argument("--codec", action="store_true",
                    help="time dequantize and validate on the full-size shapes and exit")
    ap.add_argument("--single", default=None,
                    help="run one projection of layer 0 --warmup times and exit (profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.codec:
        run_codec(args)
    elif args.prefill:
        run_prefill(args)
    elif args.single:
        run_single(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
