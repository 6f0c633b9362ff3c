"""Seeded synthetic workloads for fused sparse graph attention.

This module only draws graphs and input values. It holds none of the
attention arithmetic, so both the fp64 oracle and the CUDA path can read the
same bytes from it without sharing any computation.

Graph layout everywhere: CSR by destination.  ``row_ptr`` (int32, N+1) and
``col_idx`` (int32, E); the in-edges of destination ``i`` are
``col_idx[row_ptr[i]:row_ptr[i+1]]`` (their sources), sorted ascending.  This is
the column-pointer / row-index pair of the Triton article's CSC index
("Using the CSC index for fast edge lookup", stondelli.it/articles/gattn-triton)
and the ``row_ptr``/``col_idx`` pair of the POPCORNBENCH CSR aggregation task.

Randomness: numpy PCG64.  Graph seed = 1000 + workload number, value seed =
2000 + workload number.  Values are N(0,1) float32, cast to fp16/bf16 with
round-to-nearest-even (torch ``.to``) when the workload is a 16-bit one.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict

import numpy as np

__all__ = [
    "Graph",
    "Workload",
    "WORKLOADS",
    "tiny_poisson",
    "rtmscore_batch",
    "batched_dense",
    "powerlaw",
    "lognormal_local",
    "random_csr",
    "make_values",
    "make_workload",
]


@dataclasses.dataclass
class Graph:
    row_ptr: np.ndarray  # int32 (N+1,)
    col_idx: np.ndarray  # int32 (E,)

    @property
    def num_nodes(self) -> int:
        return int(self.row_ptr.shape[0] - 1)

    @property
    def num_edges(self) -> int:
        return int(self.col_idx.shape[0])

    def degrees(self) -> np.ndarray:
        return np.diff(self.row_ptr.astype(np.int64))


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _finish(deg: np.ndarray, col: np.ndarray) -> Graph:
    row_ptr = np.zeros(deg.shape[0] + 1, dtype=np.int64)
    np.cumsum(deg, out=row_ptr[1:])
    if row_ptr[-1] >= 2**31:
        raise ValueError("edge count does not fit int32 CSR")
    return Graph(row_ptr.astype(np.int32), np.ascontiguousarray(col.astype(np.int32)))


def _sort_within_rows(rows: np.ndarray, src: np.ndarray, n: int) -> np.ndarray:
    """Sorted source ids per destination (rows must be non-decreasing)."""
    key = rows.astype(np.int64) * n + src.astype(np.int64)
    key.sort(kind="stable")
    return (key % n).astype(np.int64)


def _dedupe_rows(rows, src, n, redraw, max_rounds=200):
    """Make sources distinct within each destination, keeping each row's count.

    ``rows`` is the non-decreasing destination of every edge; ``redraw(idx)``
    returns fresh sources for the edges at positions ``idx`` (already free of
    self loops).  Returns sources sorted ascending within every row.
    """
    key = rows.astype(np.int64) * n + src.astype(np.int64)
    key.sort()
    for _ in range(max_rounds):
        dup = np.flatnonzero(key[1:] == key[:-1]) + 1
        if dup.size == 0:
            return (key % n).astype(np.int64)
        fresh = redraw(dup)
        key[dup] = rows[dup].astype(np.int64) * n + fresh
        # re-sort only the rows that changed; positions of a row are contiguous
        bad_rows = np.unique(rows[dup])
        starts = np.searchsorted(rows, bad_rows, side="left")
        ends = np.searchsorted(rows, bad_rows, side="right")
        lens = ends - starts
        idx = np.repeat(starts - np.concatenate(([0], np.cumsum(lens)[:-1])), lens) + np.arange(lens.sum())
        key[idx] = np.sort(key[idx])
    raise RuntimeError("could not draw distinct sources")


# ---------------------------------------------------------------------------
# 1. Tiny single graph: Poisson(14) in-degree, uniform distinct sources, no
#    self loops.  N=320, 8 heads x 32, fp32 (the POPCORNBENCH task's sizes,
#    with Poisson instead of its 12..16 degrees).
# ---------------------------------------------------------------------------
def tiny_poisson(num_nodes: int = 320, mean_degree: float = 14.0, seed: int = 1001) -> Graph:
    rng = _rng(seed)
    n = num_nodes
    deg = np.minimum(rng.poisson(mean_degree, n), n - 1).astype(np.int64)
    cols = []
    for i in range(n):
        s = rng.choice(n - 1, size=int(deg[i]), replace=False)
        s = s + (s >= i)  # skip the destination itself
        cols.append(np.sort(s))
    col = np.concatenate(cols) if cols else np.zeros(0, np.int64)
    return _finish(deg, col)


# ---------------------------------------------------------------------------
# 2. RTMScore-style batch: 64 disjoint graphs of U[200,600] nodes; every node
#    has 16 in-edges from distinct nodes of its own graph (not itself).
# ---------------------------------------------------------------------------
def rtmscore_batch(num_graphs: int = 64, min_nodes: int = 200, max_nodes: int = 600,
                   in_degree: int = 16, seed: int = 1002) -> Graph:
    rng = _rng(seed)
    sizes = rng.integers(min_nodes, max_nodes + 1, num_graphs)
    degs, cols = [], []
    base = 0
    for n in sizes:
        n = int(n)
        k = min(in_degree, n - 1)
        keys = rng.random((n, n))
        np.fill_diagonal(keys, np.inf)
        pick = np.argpartition(keys, k - 1, axis=1)[:, :k] if k > 0 else np.zeros((n, 0), np.int64)
        pick.sort(axis=1)
        cols.append((pick + base).reshape(-1))
        degs.append(np.full(n, k, np.int64))
        base += n
    return _finish(np.concatenate(degs), np.concatenate(cols))


# ---------------------------------------------------------------------------
# 3. Batched dense-ish: 1024 graphs of U[20,60] nodes, directed edge
#    probability 0.3 plus self loops.
# ---------------------------------------------------------------------------
def batched_dense(num_graphs: int = 1024, min_nodes: int = 20, max_nodes: int = 60,
                  p: float = 0.3, self_loops: bool = True, seed: int = 1003) -> Graph:
    rng = _rng(seed)
    sizes = rng.integers(min_nodes, max_nodes + 1, num_graphs)
    degs, cols = [], []
    base = 0
    for n in sizes:
        n = int(n)
        adj = rng.random((n, n)) < p  # adj[dst, src]
        np.fill_diagonal(adj, self_loops)
        dst, src = np.nonzero(adj)  # row-major: grouped by dst, src ascending
        degs.append(np.bincount(dst, minlength=n).astype(np.int64))
        cols.append(src + base)
        base += n
    return _finish(np.concatenate(degs), np.concatenate(cols))


# ---------------------------------------------------------------------------
# 4. Power-law: Zipf(2.1) in-degrees truncated to [1, 10^4], rescaled by a
#    factor s (bisection) so the mean is 14; deg = clip(round(s*z), 1, 10^4).
#    Sources by preferential attachment: P(j) proportional to an independent
#    Zipf(2.1) weight per node (truncated to [1, 10^4]); distinct, not self.
# ---------------------------------------------------------------------------
def _truncated_zipf(rng, a, n, hi):
    z = rng.zipf(a, n)
    bad = np.flatnonzero(z > hi)
    while bad.size:
        z[bad] = rng.zipf(a, bad.size)
        bad = bad[z[bad] > hi]
    return z.astype(np.float64)


def powerlaw(num_nodes: int = 200_000, exponent: float = 2.1, max_degree: int = 10_000,
             mean_degree: float = 14.0, seed: int = 1004) -> Graph:
    rng = _rng(seed)
    n = num_nodes
    hi = min(max_degree, n - 1)
    z = _truncated_zipf(rng, exponent, n, max_degree)

    def degs_for(s):
        return np.clip(np.rint(s * z), 1, hi)

    lo_s, hi_s = 1e-3, float(mean_degree) * 4
    for _ in range(100):
        mid = 0.5 * (lo_s + hi_s)
        if degs_for(mid).mean() < mean_degree:
            lo_s = mid
        else:
            hi_s = mid
    deg = degs_for(0.5 * (lo_s + hi_s)).astype(np.int64)

    w = _truncated_zipf(rng, exponent, n, max_degree)
    cdf = np.cumsum(w)
    total = cdf[-1]
    rows = np.repeat(np.arange(n, dtype=np.int64), deg)

    def draw(r):
        s = np.searchsorted(cdf, rng.random(r.shape[0]) * total, side="right")
        s = np.minimum(s, n - 1)
        selfl = np.flatnonzero(s == r)
        while selfl.size:
            s2 = np.searchsorted(cdf, rng.random(selfl.size) * total, side="right")
            s[selfl] = np.minimum(s2, n - 1)
            selfl = selfl[s[selfl] == r[selfl]]
        return s

    src = draw(rows)
    col = _dedupe_rows(rows, src, n, lambda idx: draw(rows[idx]), max_rounds=100000)
    return _finish(deg, col)


# ---------------------------------------------------------------------------
# 5. Large HBM-bound: log-normal(3.6, 0.8) in-degree, deg =
#    clip(round(exp(N(3.6, 0.8^2))), 1, 20000).  60% of sources uniform in
#    [-4096, 4096]\{0} around the destination (redrawn when outside [0, N)),
#    40% uniform over all other nodes; distinct within a row.
# ---------------------------------------------------------------------------
def lognormal_local(num_nodes: int = 2_000_000, mu: float = 3.6, sigma: float = 0.8,
                    max_degree: int = 20_000, local_frac: float = 0.6, radius: int = 4096,
                    seed: int = 1005) -> Graph:
    rng = _rng(seed)
    n = num_nodes
    deg = np.clip(np.rint(np.exp(rng.normal(mu, sigma, n))), 1, min(max_degree, n - 1)).astype(np.int64)
    rows = np.repeat(np.arange(n, dtype=np.int64), deg)
    rad = min(radius, n - 1)

    def draw(r):
        m = r.shape[0]
        out = np.empty(m, np.int64)
        local = rng.random(m) < local_frac
        li = np.flatnonzero(local)
        while li.size:
            off = rng.integers(1, rad + 1, li.size) * np.where(rng.random(li.size) < 0.5, -1, 1)
            cand = r[li] + off
            ok = (cand >= 0) & (cand < n)
            out[li[ok]] = cand[ok]
            li = li[~ok]
        ui = np.flatnonzero(~local)
        s = rng.integers(0, n - 1, ui.size)
        out[ui] = s + (s >= r[ui])
        return out

    src = draw(rows)
    col = _dedupe_rows(rows, src, n, lambda idx: draw(rows[idx]), max_rounds=1000)
    return _finish(deg, col)


# ---------------------------------------------------------------------------
# Clustered heavy rows (not one of the five benchmark configurations): row
# window c (rows 16c .. 16c+15) is a community whose heavy rows each take
# `degree` distinct sources from a pool of `pool` distinct nodes shared by the
# window (uniform over all nodes); a fraction `light_frac` of the rows are
# light instead, `light_degree` distinct uniform sources from anywhere, and
# `empty_frac` of them have no entries.  The dense end of power-law graphs
# whose heavy rows cluster: windows much wider than 128 columns.
# ---------------------------------------------------------------------------
def clustered_heavy(num_windows: int = 1024, pool: int = 2048, degree: int = 1024, light_frac: float = 0.25,
                    light_degree: int = 8, empty_frac: float = 0.0, num_nodes: int = 0,
                    seed: int = 1007) -> Graph:
    rng = _rng(seed)
    n = num_nodes if num_nodes > 0 else 16 * num_windows
    degs, cols = [], []
    for w in range((n + 15) // 16):
        shared = rng.choice(n, size=min(pool, n), replace=False)
        for r in range(16 * w, min(16 * w + 16, n)):
            u = rng.random()
            if u < empty_frac:
                src = np.zeros(0, np.int64)
            elif u < empty_frac + light_frac:
                src = rng.choice(n, size=min(light_degree, n), replace=False)
            else:
                src = rng.choice(shared, size=min(degree, shared.size), replace=False)
            degs.append(src.size)
            cols.append(np.sort(src))
    return _finish(np.asarray(degs, np.int64), np.concatenate(cols) if cols else np.zeros(0, np.int64))


# ---------------------------------------------------------------------------
# Generic random CSR for edge cases (zero-degree rows, multigraphs, unsorted
# rows).  Used only by tests.
# ---------------------------------------------------------------------------
def random_csr(num_nodes: int, max_degree: int, seed: int, zero_frac: float = 0.2,
               multigraph: bool = False, sorted_rows: bool = True) -> Graph:
    rng = _rng(seed)
    n = num_nodes
    deg = rng.integers(0, max_degree + 1, n).astype(np.int64)
    deg[rng.random(n) < zero_frac] = 0
    if not multigraph:
        deg = np.minimum(deg, n)
    cols = []
    for i in range(n):
        if multigraph:
            s = rng.integers(0, n, int(deg[i]))
        else:
            s = rng.choice(n, size=int(deg[i]), replace=False)
        cols.append(np.sort(s) if sorted_rows else s)
    col = np.concatenate(cols) if cols else np.zeros(0, np.int64)
    return _finish(deg, col)


# ---------------------------------------------------------------------------
# Values
# ---------------------------------------------------------------------------
def make_values(num_nodes: int, num_edges: int, heads: int, head_dim: int,
                with_edges: bool, seed: int) -> Dict[str, np.ndarray]:
    """Q, K, V ~ N(0,1) float32 of shape (N, H, d); E (E, H, d) when asked.

    Drawn in the order Q, K, V, E from one PCG64 stream.
    """
    rng = _rng(seed)
    out = {}
    for name in ("Q", "K", "V"):
        out[name] = rng.standard_normal((num_nodes, heads, head_dim), dtype=np.float32)
    if with_edges:
        out["E"] = rng.standard_normal((num_edges, heads, head_dim), dtype=np.float32)
    return out


@dataclasses.dataclass
class Workload:
    number: int
    name: str
    graph_fn: Callable[..., Graph]
    full: dict
    small: dict
    heads: int
    head_dim: int
    dtype: str  # "f32" | "f16" | "bf16"
    variant: str  # "standard" | "rtmscore"
    description: str


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload(1, "tiny_poisson", tiny_poisson, dict(num_nodes=320), dict(num_nodes=320),
                 8, 32, "f32", "standard",
                 "N=320, Poisson(14) in-degree, uniform distinct sources, 8x32 fp32"),
        Workload(2, "rtmscore_batch64", rtmscore_batch, dict(num_graphs=64),
                 dict(num_graphs=3, min_nodes=30, max_nodes=90),
                 8, 16, "f32", "rtmscore",
                 "64 graphs of U[200,600] nodes, 16 in-edges each, 8x16 fp32, edge-modulated"),
        Workload(3, "batched_dense", batched_dense, dict(num_graphs=1024), dict(num_graphs=24),
                 8, 64, "bf16", "standard",
                 "1024 graphs of U[20,60] nodes, p=0.3 + self loops, 8x64 bf16"),
        Workload(4, "powerlaw", powerlaw, dict(num_nodes=200_000),
                 dict(num_nodes=6000, max_degree=3000),
                 1, 64, "f16", "standard",
                 "N=200k, Zipf(2.1) in-degree (mean 14, max 1e4), preferential sources, 1x64 fp16"),
        Workload(5, "lognormal_local", lognormal_local, dict(num_nodes=2_000_000),
                 dict(num_nodes=20_000, radius=1024),
                 4, 32, "bf16", "standard",
                 "N=2M, log-normal(3.6,0.8) in-degree (~100M edges), 60% sources within +-4096, 4x32 bf16"),
        # not one of the five benchmark configurations: the dense end of the
        # batched family, where the row windows are full and the tensor-core
        # tile path is the faster one (taken by default from window density 0.4)
        Workload(6, "batched_complete", batched_dense, dict(num_graphs=1024, p=1.0), dict(num_graphs=24, p=1.0),
                 8, 64, "bf16", "standard",
                 "1024 complete graphs of U[20,60] nodes (with self loops), 8x64 bf16"),
        # not one of the five either: heavy rows clustered in 16-row windows
        # (pool 2048, degree 1024), where windows are wider than the tile
        # kernel's 128 columns and run as split windows
        Workload(7, "clustered_heavy", clustered_heavy, dict(num_windows=1024),
                 dict(num_windows=12, pool=400, degree=200, empty_frac=0.05, num_nodes=187),
                 8, 64, "bf16", "standard",
                 "1024 windows of 16 rows; 3/4 of the rows take 1024 sources from a 2048-node pool shared "
                 "by the window, the rest 8 uniform sources; 8x64 bf16"),
    ]
}


def make_workload(name: str, size: str = "full", **overrides):
    """Return (graph, values_fp32, workload) for a named workload."""
    w = WORKLOADS[name]
    kw = dict(w.full if size == "full" else w.small)
    kw.update(overrides)
    kw.setdefault("seed", 1000 + w.number)
    g = w.graph_fn(**kw)
    vals = make_values(g.num_nodes, g.num_edges, w.heads, w.head_dim,
                       w.variant == "rtmscore", seed=2000 + w.number)
    return g, vals, w


def to_dtype(x: np.ndarray, dtype: str):
    """float32 numpy -> torch tensor of ``dtype`` (round-to-nearest-even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype])
