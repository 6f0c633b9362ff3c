"""Throughput benchmark of the fused sparse graph attention forward pass.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl g3s|reference]
                    [--workload lognormal_local] [--size full|small]

One step = one g3s_forward over the whole graph (fused kernel, plus the merge
of heavy-row partials), inputs resident in HBM.  The default workload is the
large HBM-bound graph: N = 2,000,000 nodes, log-normal(3.6, 0.8) in-degree
(~100.7M edges), 60% of sources within +-4096 of the destination, 4 heads x
32, bf16, standard softmax.  Its inputs (~2.5 GB touched per step) are far
larger than L2, so no explicit flush runs between steps.

Prints ONE JSON line on rank 0.  Under torchrun every rank runs its own
replica of the workload on its own GPU (independent problems, no collective
on the data path: weak scaling); time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle (the only reference this
method has) on the same workload, a bounded sample of rows per step, on the
host cores of rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import graphgen  # noqa: E402

METRIC = "edges/s of fused sparse graph attention; % of HBM or tensor-pipe roofline"
UNIT = "edges/s"
ELT = {"f32": 4, "f16": 2, "bf16": 2}
FALLBACK_HBM_GBS = 6800.0


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s)"


def measured_bf16_peak(sustained: bool):
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured (MEASURED_PEAKS.json %s)" % key
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def _strip_comments(src: str) -> str:
    """C/C++ source without comments and blank runs (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":  # literal: copy through its closing quote
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


# sources outside g3s_forward's kernels (the gather-rate probe, the projection GEMM)
NOT_FORWARD_SOURCES = ("g3s_probe.cu", "g3s_linear.cu")


def kernel_sources_hash() -> str:
    """Hash of the code of the CUDA sources g3s_forward runs (comments and
    blank lines left out, so a comment edit does not void a DRAM-traffic
    record of the same kernels)."""
    csrc = os.path.join(ROOT, "sparse_graph_attention_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".h", ".cuh")) and f not in NOT_FORWARD_SOURCES:
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode())
                h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()


def recorded_profile(workload: str):
    """ncu record of one forward on ``workload`` from profiles/traffic_<workload>.txt
    (DRAM bytes per forward, the dominant kernel and its share of device
    time), if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.txt" % workload)
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_sources_sha256") != kernel_sources_hash():
        return None
    try:
        rec = {"dram_bytes_per_forward": int(kv["dram_bytes_per_forward"])}
    except (KeyError, ValueError):
        return None
    if "dominant_kernel" in kv:
        rec["dominant_kernel"] = kv["dominant_kernel"]
    if "dominant_share" in kv:
        rec["dominant_share"] = float(kv["dominant_share"])
    return rec


def recorded_traffic(workload: str):
    """DRAM bytes per forward from the committed ncu record, if current (else None)."""
    rec = recorded_profile(workload)
    return None if rec is None else rec["dram_bytes_per_forward"]


def byte_counts(g, w, out_dtype):
    """Algorithmic bytes of one forward.

    gathered:    CSR + Q once per row + K and V once per edge (+ E in, Eout out) + O
    compulsory:  every array touched once
    """
    e, eo = ELT[w.dtype], ELT[out_dtype]
    N, E, HD = g.num_nodes, g.num_edges, w.heads * w.head_dim
    csr = 4 * (N + 1) + 4 * E
    node = N * HD * e
    out = N * HD * eo
    edge_feat = (E * HD * (e + eo)) if w.variant == "rtmscore" else 0
    gathered = csr + node + 2 * E * HD * e + edge_feat + out
    compulsory = csr + 3 * node + out + edge_feat
    return gathered, compulsory


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="g3s_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.NAMES, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Largest value of x over all ranks (the slowest rank's time); x when not distributed."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(edges_per_step: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Edges per second of all ranks together (every rank runs its own replica)."""
    return edges_per_step * steps * world / (elapsed_ms / 1000.0)


def oracle_rate(g, w, t, target_s: float, rows_start: int = 0):
    """Time the fp64 oracle on a contiguous block of rows sized for ~target_s.

    Returns (edges/s, seconds, rows, edges, threads)."""
    import oracle

    deg = g.degrees()
    args = (g.row_ptr, g.col_idx, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant, t["Q"], t["K"], t["V"],
            t.get("E"))
    # calibration on a small block
    n_cal = min(g.num_nodes, 2000)
    rows = np.arange(rows_start, rows_start + n_cal) % g.num_nodes
    t0 = time.perf_counter()
    oracle.forward(*args, rows=rows)
    dt = max(time.perf_counter() - t0, 1e-6)
    rate = deg[rows].sum() / dt
    want_edges = rate * target_s
    cum = np.cumsum(deg)
    n_rows = int(min(g.num_nodes, max(1, np.searchsorted(cum, want_edges) + 1)))
    rows = np.arange(rows_start, rows_start + n_rows) % g.num_nodes
    t0 = time.perf_counter()
    oracle.forward(*args, rows=rows)
    dt = time.perf_counter() - t0
    edges = int(deg[rows].sum())
    return edges / dt, dt, n_rows, edges, oracle.threads()


def oracle_timings(g, w, t, seconds_each: float):
    """The fp64 oracle as it stands, timed on one thread and on every core
    of this host, each on a contiguous block of rows worth ~seconds_each
    (the whole graph when it is faster)."""
    import oracle

    n_all = oracle.threads()
    out = {}
    for label, n in (("one_thread", 1), ("all_cores", n_all)):
        oracle.set_threads(n)
        rate, dt, rows, edges, _ = oracle_rate(g, w, t, seconds_each)
        out[label] = {"edges_per_s": rate, "threads": n, "seconds": dt, "rows": rows, "edges": edges}
    oracle.set_threads(n_all)
    return out


L2_FLUSH_BYTES = 256 << 20  # twice the L2 (126 MB): written between cold runs


def gather_probe_rate(dev, footprint_bytes: int, row_bytes: int, runs: int = 7, plain_loads: bool = False):
    """GB/s at which random rows of row_bytes are read from an array of about
    footprint_bytes (rounded down to a power-of-two row count; rows spread
    uniformly by multiplicative hashing; eight 512-byte warp loads in flight per
    warp, 32 warps per SM; g3s_gather_probe through the read-only path or plain
    loads), median of `runs` timed launches after two warm-ups."""
    import torch

    import sparse_graph_attention_gb300 as g3s
    rows = 2
    while rows * 2 * row_bytes <= footprint_bytes:
        rows *= 2
    src = torch.empty(rows * row_bytes // 4, dtype=torch.int32, device=dev)
    src.random_(0, 1 << 30)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas = sms * 4
    sink = torch.empty(ctas * 8, dtype=torch.int32, device=dev)
    gathers = max(1, (512 << 20) // row_bytes)  # 512 MB per launch
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        g3s.gather_probe(src, row_bytes, gathers, ctas, sink, plain_loads)
    times, n = [], 0
    for _ in range(runs):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        n = g3s.gather_probe(src, row_bytes, gathers, ctas, sink, plain_loads)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    del src, sink
    return n * row_bytes / (ms / 1e3) / 1e9


def gather_peak(dev, footprint_bytes: int, row_bytes: int) -> dict:
    """The higher of the two probe paths' rates: the random-row gather roofline
    of a footprint (the read-only path is the one the CUDA-core kernel uses)."""
    ro = gather_probe_rate(dev, footprint_bytes, row_bytes)
    pl = gather_probe_rate(dev, footprint_bytes, row_bytes, plain_loads=True)
    return {"gbs": max(ro, pl), "read_only_gbs": ro, "plain_gbs": pl}


def median_ms(step, runs: int, stream, flush=None):
    """Median over ``runs`` of one call's CUDA-event time on ``stream``; with
    ``flush`` (a device buffer larger than L2) it is overwritten before each
    run, outside the timed events, so every run starts with a cold L2."""
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
    for a, b in ev:
        if flush is not None:
            flush.add_(1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def tile_mma_flops(plan, heads: int, head_dim: int) -> int:
    """FLOPs the tile kernel issues on the tensor cores for one forward.  Per
    item (one or two windows, or one slice of a split window) and head:
    S^T = K_cols Q^T as one 128 x 16 nwin x head_dim product, and per window
    O^T = V_cols^T P^T as 128 x 16 products (the 64 feature rows issued twice)
    over its 16-column units."""
    if not plan.stats()["tile_items"]:
        return 0
    return items_mma_flops(plan.export("tile_items"), heads, head_dim)


def items_mma_flops(items, heads: int, head_dim: int) -> int:
    """The same count from an (n, 8) tile-item array."""
    items = np.asarray(items, np.int64).reshape(-1, 8)
    nwin = items[:, 3] & 0xFF
    units0 = (items[:, 3] >> 8) & 0xFF
    units1 = np.where(nwin == 2, (np.minimum(items[:, 6], 16) + 1) // 2, 0)
    per_item = 2 * 128 * 16 * nwin * head_dim + 2 * 128 * 16 * 16 * (units0 + units1)
    return int(per_item.sum() * heads)


def time_workload(name: str, dev, runs: int, oracle_seconds: float, flush, with_paths: bool):
    """One workload at full size through the default plan: warm and
    cold-L2 medians, rates, byte and FLOP fractions, the ncu record when it
    matches the sources, the oracle on one thread and on all cores; for
    the batched family and the clustered heavy rows also the CUDA-core-only
    and tile-only plans."""
    import torch

    import sparse_graph_attention_gb300 as g3s
    g, vals, w = graphgen.make_workload(name, "full")
    t = {k: graphgen.to_dtype(v, w.dtype) for k, v in vals.items()}
    rp = torch.from_numpy(g.row_ptr).to(dev)
    ci = torch.from_numpy(g.col_idx).to(dev)
    dQ, dK, dV = (t[k].to(dev) for k in "QKV")
    dE = t["E"].to(dev) if w.variant == "rtmscore" else None
    stream = torch.cuda.current_stream(dev)
    hbm, hbm_src = measured_hbm_peak()
    tf, tf_src = measured_bf16_peak(sustained=False)
    flops = 4.0 * w.heads * w.head_dim * g.num_edges

    def measure(plan):
        odt = g3s.torch_dtype(plan.out_dtype)
        O = torch.empty(dQ.shape, dtype=odt, device=dev)
        Eout = torch.empty(dE.shape, dtype=odt, device=dev) if dE is not None else None

        def step():
            if dE is not None:
                plan.forward(dQ, dK, dV, dE, O, Eout)
            else:
                plan.forward(dQ, dK, dV, None, O)

        for _ in range(5):
            step()
        torch.cuda.synchronize(dev)
        warm = median_ms(step, runs, stream)
        cold = median_ms(step, runs, stream, flush)
        plan.check()
        return warm, cold, step

    def graph_ms(step, n=20):
        """GPU time per forward inside one CUDA graph of n forwards: no host
        submission between them (the host cost of a call is timed apart)."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(n):
                step()
        for _ in range(2):
            gr.replay()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gr.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n

    def host_us(step, n=200):
        """Host time of one forward call through this binding (enqueue only)."""
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n):
            step()
        t1 = time.perf_counter()
        torch.cuda.synchronize(dev)
        return 1e6 * (t1 - t0) / n

    plan = g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant)
    st = plan.stats()
    warm, cold, step0 = measure(plan)
    in_graph = graph_ms(step0)
    call_us = host_us(step0)
    gathered, compulsory = byte_counts(g, w, plan.out_dtype)
    sec = cold / 1e3
    rec = {"num_nodes": g.num_nodes, "num_edges": g.num_edges, "heads": w.heads, "head_dim": w.head_dim,
           "dtype": w.dtype, "variant": w.variant, "out_dtype": plan.out_dtype,
           "ms_warm": warm, "ms_cold": cold, "ms_in_cuda_graph": in_graph, "host_us_per_call": call_us,
           "edges_per_s": g.num_edges / sec, "gflops": flops / sec / 1e9,
           "compulsory_frac": compulsory / sec / 1e9 / hbm, "gathered_frac": gathered / sec / 1e9 / hbm,
           "peak_gbs": hbm, "peak_source": hbm_src,
           "timing": "median of %d single-forward CUDA-event times; cold: %d MB written between runs "
                     "(outside the events) to evict L2; warm: back-to-back; in CUDA graph: one graph of 20 "
                     "forwards, GPU time per forward; host_us_per_call: the Python binding's enqueue time"
                     % (runs, L2_FLUSH_BYTES >> 20),
           "plan": {"tile_windows": st["tile_windows"], "split_windows": st["split_windows"],
                    "tile_items": st["tile_items"], "windows": st["windows"], "chunks": st["chunks"],
                    "pack_rows": st["pack_rows"], "heavy_threshold": st["heavy_threshold"],
                    "small_graph": st["small_graph"]}}
    # the gathers' own roofline: random rows of this row width over a footprint
    # the size of K and V (L2-resident here unless noted)
    row_bytes = w.heads * w.head_dim * ELT[w.dtype]
    kv_bytes = 2 * g.num_nodes * row_bytes
    peak = gather_peak(dev, kv_bytes, row_bytes)
    probe = peak["gbs"]
    gathered_rows = 2.0 * g.num_edges * row_bytes
    rec["gather_probe"] = {"row_bytes": row_bytes, "footprint_bytes": kv_bytes, "gbs": probe,
                           "read_only_gbs": peak["read_only_gbs"], "plain_gbs": peak["plain_gbs"],
                           "kv_gathers_gbs": gathered_rows / sec / 1e9,
                           "kv_gathers_frac_of_probe": gathered_rows / sec / 1e9 / probe,
                           "note": "K and V rows gathered per edge (the gathered model without CSR, Q, O, E) "
                                   "against the rate of uniform random rows of the same width over the same "
                                   "footprint"}
    prof = recorded_profile(name)
    if prof is not None:
        rec["dram_bytes"] = prof["dram_bytes_per_forward"]
        rec["dram_frac_cold"] = prof["dram_bytes_per_forward"] / sec / 1e9 / hbm
        if "dominant_kernel" in prof:
            rec["dominant_kernel"] = prof["dominant_kernel"]
            rec["dominant_share"] = prof.get("dominant_share")
    if st["tile_windows"] > 0:
        issued = tile_mma_flops(plan, w.heads, w.head_dim)
        useful = 4.0 * w.heads * w.head_dim * st["tile_window_nnz"]
        rec["tile"] = {"useful_flops": useful, "issued_flops": issued,
                       "useful_frac_of_forward": useful / sec / 1e12 / tf,
                       "peak_tflops": tf, "peak_source": tf_src + " (fp16 dense rate equals bf16's)"}
    if with_paths:
        paths = {}
        for label, kw in (("core_only", dict(tile_path=0)),
                          ("tile_only", dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0))):
            p2 = g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant, **kw)
            s2 = p2.stats()
            w2, c2, _ = measure(p2)
            entry = {"ms_warm": w2, "ms_cold": c2, "tile_windows": s2["tile_windows"],
                     "split_windows": s2["split_windows"], "windows": s2["windows"]}
            if s2["tile_windows"] > 0:
                useful = 4.0 * w.heads * w.head_dim * s2["tile_window_nnz"]
                issued = tile_mma_flops(p2, w.heads, w.head_dim)
                entry["tile_useful_tflops"] = useful / (c2 / 1e3) / 1e12
                entry["tile_useful_frac"] = entry["tile_useful_tflops"] / tf
                entry["tile_issued_frac"] = issued / (c2 / 1e3) / 1e12 / tf
                entry["tile_window_nnz"] = s2["tile_window_nnz"]
            paths[label] = entry
            p2.close()
        rec["paths"] = paths
    if oracle_seconds > 0:
        rec["oracle"] = oracle_timings(g, w, t, oracle_seconds)
    plan.close()
    del dQ, dK, dV, dE, rp, ci
    torch.cuda.empty_cache()
    return rec


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["g3s", "reference"], default="g3s")
    ap.add_argument("--workload", default="lognormal_local", choices=list(graphgen.WORKLOADS))
    ap.add_argument("--size", default="full", choices=["full", "small"])
    ap.add_argument("--nodes", type=int, default=None, help="override the workload's node count (profiling)")
    ap.add_argument("--local-frac", type=float, default=None,
                    help="lognormal_local only: override the share of sources within +-4096 rows (default 0.6; "
                         "1.0 and 0.0 separate the L2-served gathers from the HBM-served ones)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle work for the cpu_baseline sample")
    ap.add_argument("--tile-path", type=int, default=-1, choices=[-1, 0, 1],
                    help="tensor-core tile path: -1 automatic (default), 0 off, 1 on")
    ap.add_argument("--tile-density-milli", type=int, default=None,
                    help="density cutoff of the tile path in 1/1000 (default: the library's)")
    ap.add_argument("--tile-pool-density-milli", type=int, default=None,
                    help="pooled density the tile-eligible windows need to take the tile path (default: the library's)")
    ap.add_argument("--tile-split-parallel", type=int, default=None, choices=[0, 1],
                    help="split windows (wider than 128 columns): 0 node-parallel chains, 1 edge-parallel slices "
                         "merged (default: the library's)")
    ap.add_argument("--out-dtype", default=None, choices=["f32", "f16", "bf16"],
                    help="element type of O (default fp32)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the forward captured in a CUDA graph (no per-call launch overhead)")
    ap.add_argument("--layer", type=int, default=0, metavar="KIN",
                    help="also time one attention layer on 16-bit workloads: Q|K|V = X Wqkv^T for X of KIN "
                         "features (the tcgen05 projection), then the forward; adds a 'layer' object")
    ap.add_argument("--aggregate", action="store_true",
                    help="also time g3s_aggregate (normalised weighted aggregation) on the workload's graph; "
                         "adds an 'aggregate' object")
    ap.add_argument("--pack-rows", type=int, default=None, choices=[0, 1],
                    help="short-row packs, one row per lane group (default: the library's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="plans (each with its own staging) taking e2e steps in turn, one stream each")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gather-probe", action="store_true",
                    help="only run the gather-rate probe over a range of footprints and row widths; print JSON")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the 'workloads' record (the other benchmark graphs, timed warm and cold)")
    ap.add_argument("--workload-runs", type=int, default=20, help="timed runs per workload (median)")
    ap.add_argument("--workload-oracle-seconds", type=float, default=1.5,
                    help="oracle work per workload and thread count")
    return ap.parse_args()


def run_reference(args, rank):
    if rank != 0:
        return
    g, vals, w = graphgen.make_workload(args.workload, args.size)
    t = {k: graphgen.to_dtype(v, w.dtype) for k, v in vals.items()}
    per_step = max(0.2, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    start = 0
    for _ in range(args.warmup):
        _, _, n, _, _ = oracle_rate(g, w, t, per_step, start)
        start = (start + n) % g.num_nodes
    total_edges, total_s, threads = 0, 0.0, 1
    for _ in range(args.steps):
        _, dt, n, edges, threads = oracle_rate(g, w, t, per_step, start)
        start = (start + n) % g.num_nodes
        total_edges += edges
        total_s += dt
    value = total_edges / total_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "num_nodes": g.num_nodes, "num_edges": g.num_edges, "heads": w.heads,
                   "head_dim": w.head_dim, "input_dtype": w.dtype, "variant": w.variant},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "per step a contiguous block of rows (~%.1f s of fp64 oracle work), "
                                   "%d edges over %d steps" % (per_step, total_edges, args.steps)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def aggregate_bytes(g, w, out_dtype):
    """Algorithmic bytes of one g3s_aggregate: CSR + per edge its weights (H)
    and its source row of X (H*d) + O written once; the compulsory count
    reads X once instead of once per edge."""
    e, eo = ELT[w.dtype], ELT[out_dtype]
    N, E, H, HD = g.num_nodes, g.num_edges, w.heads, w.heads * w.head_dim
    csr = 4 * (N + 1) + 4 * E
    gathered = csr + E * H * e + E * HD * e + N * HD * eo
    compulsory = csr + E * H * e + N * HD * e + N * HD * eo
    return gathered, compulsory


def time_aggregate(args, g, w, plan, O, stream, dev):
    """g3s_aggregate (normalised weighted aggregation) over the workload's
    graph, X = the workload's V, seeded positive weights per edge and head."""
    import torch
    import sparse_graph_attention_gb300 as g3s
    tdt = g3s.torch_dtype(w.dtype)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4000 + w.number)
    X = torch.randn(g.num_nodes, w.heads, w.head_dim, device=dev, generator=gen).to(tdt)
    Wt = (torch.rand(g.num_edges, w.heads, device=dev, generator=gen) + 0.05).to(tdt)

    def step():
        plan.aggregate(Wt, X, O=O, normalize=True, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 100))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / n
    gathered, compulsory = aggregate_bytes(g, w, plan.out_dtype)
    hbm, hbm_src = measured_hbm_peak()
    sec = ms / 1e3
    return {"ms": ms, "edges_per_s": g.num_edges / sec, "normalize": True,
            "roofline": {"bound": "hbm", "achieved": gathered / sec / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": gathered / sec / 1e9 / hbm, "peak_source": hbm_src,
                         "compulsory_gbs": compulsory / sec / 1e9, "compulsory_frac": compulsory / sec / 1e9 / hbm,
                         "bytes_model": "gathered: CSR + W per edge + X row per edge + O; compulsory: X once"},
            "data": "seeded synthetic X and positive weights (torch generator)"}


def time_layer(args, g, w, plan, O, Eout, stream, dev):
    """One attention layer: Q|K|V = X Wqkv^T (g3s_linear, tensor cores) then the
    fused forward, on seeded synthetic features and weights of the workload's
    shape; the projection alone is timed too and set against its roofline."""
    import torch
    import sparse_graph_attention_gb300 as g3s
    if w.dtype not in ("bf16", "f16"):
        return {"unavailable": "the projection takes 16-bit inputs; this workload is %s" % w.dtype}
    kin = int(args.layer)
    hd = w.heads * w.head_dim
    tdt = g3s.torch_dtype(w.dtype)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000 + w.number)
    X = torch.randn(g.num_nodes, kin, device=dev, generator=gen).to(tdt)
    Wqkv = (torch.randn(3 * hd, kin, device=dev, generator=gen) * kin ** -0.5).to(tdt)
    Xe = We = None
    if w.variant == "rtmscore":
        Xe = torch.randn(g.num_edges, kin, device=dev, generator=gen).to(tdt)
        We = (torch.randn(hd, kin, device=dev, generator=gen) * kin ** -0.5).to(tdt)
    qkv = [torch.empty(g.num_nodes, hd, dtype=tdt, device=dev) for _ in range(3)]

    def layer_step():
        plan.layer_forward(X, Wqkv, Xe, We, O=O, Eout=Eout)

    def proj_step():
        g3s.linear(X, Wqkv, seg_cols=hd, outs=qkv, stream=stream)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n

    n = max(3, min(args.steps, 50))
    layer_ms = timed(layer_step, n)
    proj_ms = timed(proj_step, n)
    flops = 2.0 * g.num_nodes * kin * 3 * hd
    nbytes = 2.0 * (g.num_nodes * kin + 3 * hd * kin + g.num_nodes * 3 * hd)
    hbm, hbm_src = measured_hbm_peak()
    tf, tf_src = measured_bf16_peak(sustained=False)
    if w.dtype == "f16":
        tf_src += " (fp16 dense rate equals bf16's)"
    t_mem, t_math = nbytes / (hbm * 1e9), flops / (tf * 1e12)
    if t_mem >= t_math:
        roof = {"bound": "hbm", "achieved": nbytes / (proj_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                "peak_source": hbm_src}
    else:
        roof = {"bound": "tensor", "achieved": flops / (proj_ms / 1e3) / 1e12, "peak": tf, "unit": "TFLOP/s",
                "peak_source": tf_src}
    roof["frac"] = roof["achieved"] / roof["peak"]
    return {"kin": kin, "ms_per_layer": layer_ms, "edges_per_s": g.num_edges / (layer_ms / 1e3),
            "projection": {"ms": proj_ms, "shape": [g.num_nodes, kin, 3 * hd], "tflops": flops / (proj_ms / 1e3) / 1e12,
                           "gbs": nbytes / (proj_ms / 1e3) / 1e9, "roofline": roof,
                           "bytes_model": "X read once, Wqkv once, Q|K|V written once (16-bit)"},
            "data": "seeded synthetic features and weights (torch generator), not trained"}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch

    import sparse_graph_attention_gb300 as g3s

    if args.gather_probe:
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        res = []
        for footprint in (16 << 20, 32 << 20, 64 << 20, 128 << 20, 256 << 20, 1 << 30):
            for rb in (128, 256, 512, 1024):
                res.append(dict(gather_peak(dev, footprint, rb), footprint_mb=footprint >> 20, row_bytes=rb))
        print(json.dumps({"gather_probe": res}), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    over = {} if args.nodes is None else {"num_nodes": args.nodes}
    if args.local_frac is not None:
        if args.workload != "lognormal_local":
            raise SystemExit("--local-frac applies to the lognormal_local workload")
        over["local_frac"] = args.local_frac
    g, vals, w = graphgen.make_workload(args.workload, args.size, **over)
    t = {k: graphgen.to_dtype(v, w.dtype) for k, v in vals.items()}
    rp = torch.from_numpy(g.row_ptr).to(dev)
    ci = torch.from_numpy(g.col_idx).to(dev)
    dQ, dK, dV = (t[k].to(dev) for k in "QKV")
    dE = t["E"].to(dev) if w.variant == "rtmscore" else None
    stream = torch.cuda.current_stream(dev)

    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    plan_kw = {"tile_path": args.tile_path}
    if args.out_dtype:
        plan_kw["out_dtype"] = args.out_dtype
    if args.tile_density_milli is not None:
        plan_kw["tile_density_milli"] = args.tile_density_milli
    if args.tile_pool_density_milli is not None:
        plan_kw["tile_pool_density_milli"] = args.tile_pool_density_milli
    if args.tile_split_parallel is not None:
        plan_kw["tile_split_parallel"] = args.tile_split_parallel
    if args.pack_rows is not None:
        plan_kw["pack_rows"] = args.pack_rows
    plan = g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant, **plan_kw)
    torch.cuda.synchronize(dev)
    plan_ms = 1000.0 * (time.perf_counter() - t0)
    st = plan.stats()
    launches = 1 + (1 if st["chunks"] > 0 else 0) + (1 if st["tile_windows"] > 0 else 0)

    odt = g3s.torch_dtype(plan.out_dtype)
    O = torch.empty(dQ.shape, dtype=odt, device=dev)
    Eout = torch.empty(dE.shape, dtype=odt, device=dev) if dE is not None else None

    def step():
        if w.variant == "rtmscore":
            plan.forward(dQ, dK, dV, dE, O, Eout)
        else:
            plan.forward(dQ, dK, dV, None, O)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if args.graph:  # capture one forward, then time replays of it
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream(dev).wait_stream(side)
        fwd_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fwd_graph):
            step()
        step = fwd_graph.replay
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)

    # ---- timed region: K forwards, inputs resident ----------------------
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank)
    time.sleep(0.3)  # let the sampler start before the work does
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if dist:
        dist.barrier()
    total_ms = t_all0.elapsed_time(t_all1)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(g.num_edges, args.steps, world, total_ms)

    # ---- roofline of the forward (fused kernel + heavy-row merge) --------
    # frac: DRAM bytes one forward moves (ncu, recorded on these kernel
    # sources) / the live mean launch time / the measured copy peak.  The
    # gathered-bytes model (every K, V row read once per edge) exceeds the
    # DRAM bytes where sources repeat in L2, so its fraction is kept beside
    # it as gathered_frac, with the compulsory lower bound (every array once).
    gathered, compulsory = byte_counts(g, w, plan.out_dtype)
    fwd_s = statistics.mean(per_launch_ms) / 1000.0
    peak, peak_src = measured_hbm_peak()
    prof = recorded_profile(w.name)
    traffic = None if prof is None else prof["dram_bytes_per_forward"]
    basis = traffic if traffic is not None else compulsory
    achieved = basis / fwd_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_source": peak_src,
                "basis": ("ncu DRAM bytes per forward (dram__bytes_read.sum + dram__bytes_write.sum, "
                          "profiles/traffic_%s.txt, same kernel sources) / live mean forward time" % w.name)
                if traffic is not None else
                "compulsory bytes (no ncu DRAM record for the current kernel sources): a lower bound",
                "kernel": "g3s_forward (fused CUDA-core kernel + heavy-row merge)",
                "gathered_gbs": gathered / fwd_s / 1e9, "gathered_frac": gathered / fwd_s / 1e9 / peak,
                "bytes_model": "gathered: CSR + Q + K,V per edge (+E, Eout) + O (L2 hits of local sources let "
                               "it exceed 1); compulsory: every array once",
                "compulsory_gbs": compulsory / fwd_s / 1e9,
                "compulsory_frac": compulsory / fwd_s / 1e9 / peak}
    if prof is not None and "dominant_kernel" in prof:
        roofline["dominant_kernel"] = prof["dominant_kernel"]
        roofline["dominant_share"] = prof.get("dominant_share")
    if not args.no_workloads:
        rb = w.heads * w.head_dim * ELT[w.dtype]
        rate = gather_peak(dev, 2 * g.num_nodes * rb, rb)["gbs"]
        roofline["random_row_gather_gbs"] = rate
        roofline["random_row_gather_note"] = ("uniform random %d-byte rows over the %.2f GB K+V footprint "
                                             "(g3s_gather_probe): the rate the 40%% non-local gathers can be "
                                             "served at" % (rb, 2 * g.num_nodes * rb / 1e9))

    # ---- optional: a whole layer (projection on the tensor cores + forward) ----
    layer = None
    if args.layer:
        layer = time_layer(args, g, w, plan, O, Eout, stream, dev)
    aggregate = None
    if args.aggregate:
        aggregate = time_aggregate(args, g, w, plan, O, stream, dev)

    # ---- end to end through the C ABI on host buffers --------------------
    # Every step uploads its Q, K, V (and E) from pinned host memory and
    # downloads its O (and Eout) through g3s_forward_host.  Three plans (each
    # with its own workspace and device staging) take the steps in turn, one
    # stream each, so one step's upload overlaps the others' kernels and
    # downloads, as a caller streaming feature batches over one graph would
    # run it (with two, a stream's next upload waited behind its own
    # download).  The serialised single-stream time is reported beside it.
    e2e = None
    if not args.no_e2e:
        pin = {k: t[k].pin_memory() for k in t}
        ns = max(1, args.e2e_streams)
        plans = [plan] + [g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant, **plan_kw)
                          for _ in range(ns - 1)]
        streams = [torch.cuda.Stream(dev) for _ in range(ns)]
        stagings = [torch.empty(pl.staging_size(), dtype=torch.uint8, device=dev) for pl in plans]
        Ohs = [torch.empty(pin["Q"].shape, dtype=odt).pin_memory() for _ in range(ns)]
        Eohs = [torch.empty(pin["E"].shape, dtype=odt).pin_memory() if w.variant == "rtmscore" else None
                for _ in range(ns)]

        def host_step(i, k=None):
            k = i % ns if k is None else k
            plans[k].forward_host(pin["Q"], pin["K"], pin["V"], Ohs[k], pin.get("E"), Eohs[k], staging=stagings[k],
                                  stream=streams[k])

        def timed(n, pipelined):
            main = torch.cuda.current_stream(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for st_ in streams:
                st_.wait_event(a)
            for i in range(n):
                host_step(i, None if pipelined else 0)
            for st_ in streams:
                ev = torch.cuda.Event()
                ev.record(st_)
                main.wait_event(ev)
            b.record(main)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b)

        for i in range(4):
            host_step(i)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        n_e2e = max(2, min(args.steps, 50))
        e2e_ms = max_over_ranks(timed(n_e2e, True), dist, dev)
        serial_ms = max_over_ranks(timed(max(1, n_e2e // 5), False), dist, dev) / max(1, n_e2e // 5)
        hd = w.heads * w.head_dim
        nb, nbo = g.num_nodes * hd * ELT[w.dtype], g.num_nodes * hd * ELT[plan.out_dtype]
        eb, ebo = g.num_edges * hd * ELT[w.dtype], g.num_edges * hd * ELT[plan.out_dtype]
        h2d = 3 * nb + (eb if w.variant == "rtmscore" else 0)
        d2h = nbo + (ebo if w.variant == "rtmscore" else 0)
        e2e = {"value": whole_job_rate(g.num_edges, n_e2e, world, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": e2e_ms / n_e2e, "serial_ms_per_step": serial_ms,
               "path": "g3s_forward_host, pinned host buffers, %d plans in turn on %d streams" % (ns, ns)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, dt, n_rows, edges, threads = oracle_rate(g, w, t, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "rows 0..%d (%d edges, %.1f s) of the same workload, fp64 oracle" % (n_rows - 1, edges, dt)}
        import oracle
        oracle.set_threads(1)
        r1, dt1, n1, e1, _ = oracle_rate(g, w, t, args.cpu_seconds / 4)
        oracle.set_threads(threads)
        cpu["one_thread"] = {"value": r1, "cores": 1,
                             "sample": "rows 0..%d (%d edges, %.1f s)" % (n1 - 1, e1, dt1)}

    # ---- the other workloads (rank 0): each at full size, warm and cold L2 ----
    workloads = None
    if rank == 0 and not args.no_workloads:
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        workloads = {}
        for name in ("tiny_poisson", "rtmscore_batch64", "batched_dense", "powerlaw", "batched_complete",
                     "clustered_heavy"):
            workloads[name] = time_workload(name, dev, args.workload_runs,
                                            0.0 if args.no_cpu_baseline else args.workload_oracle_seconds, flush,
                                            with_paths=name.startswith("batched") or name == "clustered_heavy")
        del flush

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "description": w.description, "num_nodes": g.num_nodes,
                       "num_edges": g.num_edges, "heads": w.heads, "head_dim": w.head_dim, "variant": w.variant,
                       "out_dtype": plan.out_dtype, "accumulation": "f32",
                       "l2": "no flush: inputs larger than L2 (%.2f GB touched per step)" % (compulsory / 1e9),
                       "parallelism": "replica per GPU" if world > 1 else "single GPU",
                       "launch": "CUDA graph replay" if args.graph else "one g3s_forward call per step"},
            "gflops": 4.0 * w.heads * w.head_dim * g.num_edges / (ms_per_step / 1000.0) / 1e9,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches * args.steps, "clocks": clocks, "plan_ms": plan_ms, "layer": layer,
            "aggregate": aggregate, "workloads": workloads,
            "plan": {"heavy_rows": st["heavy_rows"], "chunks": st["chunks"],
                     "heavy_threshold": st["heavy_threshold"], "pack_rows": st["pack_rows"],
                     "tile_windows": st["tile_windows"],
                     "tiles": st["tiles"], "tile_window_nnz": st["tile_window_nnz"]},
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
