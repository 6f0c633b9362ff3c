"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` function takes ``fwd``, a callable with the signature of
``oracle.forward``, and raises ``AssertionError`` when the oracle disagrees
with what the pages and the mathematics fix.  ``test_oracle_pins.py`` runs them
on the real oracle; ``test_oracle_mutants.py`` runs them on copies of the
oracle with planted mistakes and requires that every mistake is caught.

Nothing here calls the CUDA library.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS = 1e-6


def _csr_from_pairs(n, pairs):
    pairs = sorted(pairs)
    deg = np.zeros(n, np.int64)
    for dst, _ in pairs:
        deg[dst] += 1
    row_ptr = np.zeros(n + 1, np.int32)
    row_ptr[1:] = np.cumsum(deg)
    col = np.array([s for _, s in pairs], np.int32)
    return row_ptr, col


def four_node():
    with open(os.path.join(GOLDEN, "four_node_example.json")) as f:
        g = json.load(f)
    pairs = [tuple(p) for p in g["edges_dst_src"]]
    row_ptr, col = _csr_from_pairs(4, pairs)
    q = np.array(g["q"], np.float32).reshape(4, 1, 4)
    k = np.array(g["k"], np.float32).reshape(4, 1, 4)
    v = np.array(g["v"], np.float32).reshape(4, 1, 4)
    ordered = sorted(pairs)
    e = np.array([g["e_override"].get("%d<-%d" % p, g["e_default"]) for p in ordered],
                 np.float32).reshape(-1, 1, 4)
    return row_ptr, col, q, k, v, e, ordered


# ---------------------------------------------------------------------------
# 1. The hand-worked example: closed forms
# ---------------------------------------------------------------------------
def pin_four_node_standard(fwd):
    row_ptr, col, q, k, v, _, _ = four_node()
    O = fwd(row_ptr, col, 4, 1, 4, "f32", "standard", q, k, v)[:, 0, :]
    e = math.e
    # row 0: logits <q0,k1>/2 = 1 and <q0,k2>/2 = 0
    exp0 = np.array([e / (1 + e), 1 / (1 + e), 0, 0])
    # row 1: logits 0 (k0 = 0) and <q1,k3>/2 = 15/2
    w3 = math.exp(7.5) / (1 + math.exp(7.5))
    exp1 = np.array([0, 0, 1 - w3, w3])
    # row 2: q2 = 0, uniform over sources 0, 1, 3
    exp2 = np.array([1 / 3, 0, 1 / 3, 1 / 3])
    exp3 = np.zeros(4)  # no in-edges
    want = np.stack([exp0, exp1, exp2, exp3])
    assert np.allclose(O, want, rtol=0, atol=1e-14), (O, want)


def pin_four_node_rtmscore(fwd):
    row_ptr, col, q, k, v, ev, ordered = four_node()
    O, Eout = fwd(row_ptr, col, 4, 1, 4, "f32", "rtmscore", q, k, v, ev, want_eout=True)
    O = O[:, 0, :]
    e = math.e
    d0 = e + 1 + EPS
    exp0 = np.array([e / d0, 1 / d0, 0, 0])
    # row 1, page order: clamp(5*3/2) = 5 elementwise, times 0.5 -> logit 2.5
    s13 = math.exp(2.5)
    d1 = 1 + s13 + EPS
    exp1 = np.array([0, 0, 1 / d1, s13 / d1])
    d2 = 3 + EPS
    exp2 = np.array([1 / d2, 0, 1 / d2, 1 / d2])
    want = np.stack([exp0, exp1, exp2, np.zeros(4)])
    assert np.allclose(O, want, rtol=0, atol=1e-14), (O, want)
    pos = {p: i for i, p in enumerate(ordered)}
    assert np.allclose(Eout[pos[(0, 1)], 0], [1, 0, 0, 0], atol=0)
    assert np.allclose(Eout[pos[(1, 3)], 0], [2.5, 0, 0, 0], atol=0)
    assert np.allclose(Eout[pos[(1, 0)], 0], [0, 0, 0, 0], atol=0)
    # the literal order (no elementwise clamp): logit 15/2 * 0.5 = 3.75
    O2 = fwd(row_ptr, col, 4, 1, 4, "f32", "rtmscore", q, k, v, ev, elementwise_clamp=False)[:, 0, :]
    s13b = math.exp(3.75)
    d1b = 1 + s13b + EPS
    assert np.allclose(O2[1], [0, 0, 1 / d1b, s13b / d1b], rtol=0, atol=1e-14)
    assert np.allclose(O2[0], exp0, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# 2. Brute force: dense masked attention on small graphs
# ---------------------------------------------------------------------------
def dense_standard(row_ptr, col, n, q, k, v):
    """Dense masked softmax attention with edge multiplicities, fp64."""
    H, d = q.shape[1], q.shape[2]
    C = np.zeros((n, n))
    for i in range(n):
        for e in range(row_ptr[i], row_ptr[i + 1]):
            C[i, col[e]] += 1
    out = np.zeros((n, H, d))
    for h in range(H):
        S = q[:, h, :].astype(np.float64) @ k[:, h, :].astype(np.float64).T / math.sqrt(d)
        S = np.where(C > 0, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        P = C * np.exp(S - m)
        den = P.sum(axis=1, keepdims=True)
        num = P @ v[:, h, :].astype(np.float64)
        out[:, h, :] = np.where(den > 0, num / np.where(den > 0, den, 1), 0.0)
    return out


def dense_rtmscore(row_ptr, col, n, q, k, v, e, elementwise_clamp=True):
    """Dense form of the edge-modulated variant on a simple graph, fp64."""
    H, d = q.shape[1], q.shape[2]
    mask = np.zeros((n, n), bool)
    Ed = np.zeros((n, n, H, d))
    for i in range(n):
        for x in range(row_ptr[i], row_ptr[i + 1]):
            mask[i, col[x]] = True
            Ed[i, col[x]] = e[x]
    q64, k64, v64 = (a.astype(np.float64) for a in (q, k, v))
    T = q64[:, None, :, :] * k64[None, :, :, :] / math.sqrt(d)  # (dst, src, H, d)
    if elementwise_clamp:
        T = np.clip(T, -5, 5)
    U = T * Ed
    L = np.clip(U.sum(-1), -5, 5)  # (dst, src, H)
    S = np.where(mask[:, :, None], np.exp(L), 0.0)
    num = np.einsum("ijh,jhf->ihf", S, v64)
    den = S.sum(axis=1)[:, :, None] + EPS
    eout = np.zeros((col.size, H, d))
    for i in range(n):
        for x in range(row_ptr[i], row_ptr[i + 1]):
            eout[x] = U[i, col[x]]
    return num / den, eout


def _rand_graph(seed, n, maxdeg, multigraph):
    import graphgen

    g = graphgen.random_csr(n, maxdeg, seed=seed, zero_frac=0.25, multigraph=multigraph,
                            sorted_rows=False)
    return g.row_ptr, g.col_idx


def pin_brute_force_standard(fwd):
    for seed, (n, H, d, maxdeg, multi) in enumerate([(40, 2, 8, 12, False), (33, 3, 16, 20, True),
                                                      (64, 1, 4, 64, False), (17, 4, 32, 5, True)]):
        rng = np.random.default_rng(100 + seed)
        rp, col = _rand_graph(200 + seed, n, maxdeg, multi)
        q, k, v = (rng.standard_normal((n, H, d)).astype(np.float32) for _ in range(3))
        got = fwd(rp, col, n, H, d, "f32", "standard", q, k, v)
        want = dense_standard(rp, col, n, q, k, v)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), np.abs(got - want).max()


def pin_brute_force_rtmscore(fwd):
    for seed, (n, H, d, maxdeg, scale) in enumerate([(30, 2, 8, 10, 1.0), (25, 3, 16, 25, 4.0),
                                                      (12, 1, 4, 12, 12.0)]):
        rng = np.random.default_rng(300 + seed)
        rp, col = _rand_graph(400 + seed, n, maxdeg, False)
        q, k, v = (rng.standard_normal((n, H, d)).astype(np.float32) * s
                   for s in (scale, scale, 1.0))
        e = rng.standard_normal((col.size, H, d)).astype(np.float32)
        for ec in (True, False):
            got, gout = fwd(rp, col, n, H, d, "f32", "rtmscore", q, k, v, e, want_eout=True,
                            elementwise_clamp=ec)
            want, wout = dense_rtmscore(rp, col, n, q, k, v, e, elementwise_clamp=ec)
            assert np.allclose(got, want, rtol=1e-12, atol=1e-12), np.abs(got - want).max()
            assert np.allclose(gout, wout, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# 3. Invariants and closed forms
# ---------------------------------------------------------------------------
def _graph_and_values(seed, n=50, H=2, d=16, maxdeg=15, with_e=False):
    rng = np.random.default_rng(seed)
    rp, col = _rand_graph(seed + 7, n, maxdeg, False)
    q, k, v = (rng.standard_normal((n, H, d)).astype(np.float32) for _ in range(3))
    e = rng.standard_normal((col.size, H, d)).astype(np.float32) if with_e else None
    return rp, col, q, k, v, e


def pin_permutation_invariance(fwd):
    for variant in ("standard", "rtmscore"):
        rp, col, q, k, v, e = _graph_and_values(11, with_e=True)
        n, H, d = q.shape
        rng = np.random.default_rng(5)
        perm = np.arange(col.size)
        for i in range(n):
            a, b = rp[i], rp[i + 1]
            perm[a:b] = a + rng.permutation(b - a)
        O1 = fwd(rp, col, n, H, d, "f32", variant, q, k, v, e)
        O2 = fwd(rp, col[perm], n, H, d, "f32", variant, q, k, v, e[perm])
        assert np.allclose(O1, O2, rtol=1e-13, atol=1e-14)


def pin_zero_degree_and_weights(fwd):
    rp, col, q, k, v, e = _graph_and_values(21, with_e=True)
    n, H, d = q.shape
    deg = np.diff(rp)
    assert (deg == 0).any() and (deg > 0).any()
    ones = np.ones_like(v)
    # standard: weights sum to one -> O = 1 on rows with in-edges
    O = fwd(rp, col, n, H, d, "f32", "standard", q, k, ones)
    assert np.allclose(O[deg > 0], 1.0, rtol=0, atol=1e-14)
    assert np.all(O[deg == 0] == 0.0)
    # variant: weights sum to S/(S+eps) with S in [deg e^-5, deg e^5]
    O = fwd(rp, col, n, H, d, "f32", "rtmscore", q, k, ones, e)
    assert np.all(O[deg == 0] == 0.0)
    dd = deg[deg > 0][:, None, None].astype(np.float64)
    lo = dd * math.exp(-5) / (dd * math.exp(-5) + EPS)
    hi = dd * math.exp(5) / (dd * math.exp(5) + EPS)
    Ov = O[deg > 0]
    assert np.all(Ov >= lo - 1e-15) and np.all(Ov <= hi + 1e-15) and np.all(Ov < 1.0)


def pin_convex_hull(fwd):
    rp, col, q, k, v, _ = _graph_and_values(31)
    n, H, d = q.shape
    O = fwd(rp, col, n, H, d, "f32", "standard", q * 3, k * 3, v)
    for i in range(n):
        srcs = col[rp[i]:rp[i + 1]]
        if srcs.size == 0:
            continue
        lo = v[srcs].min(axis=0)
        hi = v[srcs].max(axis=0)
        assert np.all(O[i] >= lo - 1e-12) and np.all(O[i] <= hi + 1e-12)


def pin_closed_forms(fwd):
    rp, col, q, k, v, e = _graph_and_values(41, with_e=True)
    n, H, d = q.shape
    deg = np.diff(rp)
    zq = np.zeros_like(q)
    mean = np.zeros((n, H, d))
    sums = np.zeros((n, H, d))
    for i in range(n):
        srcs = col[rp[i]:rp[i + 1]]
        if srcs.size:
            sums[i] = v[srcs].astype(np.float64).sum(axis=0)
            mean[i] = sums[i] / srcs.size
    # Q = 0: uniform logits -> mean of neighbours (standard), sum/(deg+eps) (variant)
    O = fwd(rp, col, n, H, d, "f32", "standard", zq, k, v)
    assert np.allclose(O, mean, rtol=1e-13, atol=1e-14)
    O = fwd(rp, col, n, H, d, "f32", "rtmscore", zq, k, v, e)
    want = sums / (deg[:, None, None] + EPS)
    assert np.allclose(O, want, rtol=1e-13, atol=1e-14)
    # a single in-edge: O = v_j (standard)
    rp1 = np.arange(n + 1, dtype=np.int32)
    col1 = ((np.arange(n) * 7 + 3) % n).astype(np.int32)
    O = fwd(rp1, col1, n, H, d, "f32", "standard", q, k, v)
    assert np.allclose(O, v[col1].astype(np.float64), rtol=0, atol=1e-15)


def pin_clip_bounds(fwd):
    rp, col, q, k, v, e = _graph_and_values(51, with_e=True)
    n, H, d = q.shape
    _, Eout = fwd(rp, col, n, H, d, "f32", "rtmscore", q * 8, k * 8, v, e, want_eout=True)
    assert np.all(np.abs(Eout) <= 5 * np.abs(e.astype(np.float64)) + 1e-12)
    assert np.any(np.abs(Eout) >= 5 * np.abs(e.astype(np.float64)) - 1e-12)  # clamp reached


def pin_library_softmax(fwd):
    """Complete bipartite block: every row sees every node -> torch softmax(QK^T/sqrt d) V."""
    import torch

    n, H, d = 24, 3, 16
    rng = np.random.default_rng(61)
    q, k, v = (rng.standard_normal((n, H, d)).astype(np.float32) for _ in range(3))
    rp = (np.arange(n + 1) * n).astype(np.int32)
    col = np.tile(np.arange(n), n).astype(np.int32)
    O = fwd(rp, col, n, H, d, "f32", "standard", q, k, v)
    qt, kt, vt = (torch.from_numpy(a).double().transpose(0, 1) for a in (q, k, v))
    ref = torch.softmax(qt @ kt.transpose(1, 2) / math.sqrt(d), dim=-1) @ vt
    assert np.allclose(O, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-13)


def pin_sixteen_bit_inputs(fwd):
    """16-bit inputs are read exactly: same answer as fp32 arrays holding the same values."""
    import torch

    rp, col, q, k, v, e = _graph_and_values(71, with_e=True)
    n, H, d = q.shape
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        t = [torch.from_numpy(a).to(tdt) for a in (q, k, v, e)]
        wide = [x.float().numpy() for x in t]
        for variant in ("standard", "rtmscore"):
            got = fwd(rp, col, n, H, d, dt, variant, *t)
            want = fwd(rp, col, n, H, d, "f32", variant, *wide)
            assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# 4. Weighted aggregation
# ---------------------------------------------------------------------------
def pin_aggregate_reference_loop(agg):
    """The CSR aggregation task's reference loop: out[dst] = (x[src] * w[start:end, :, None]).sum(0)."""
    for seed, (n, H, d, multi) in enumerate([(40, 8, 32, False), (33, 2, 16, True), (17, 1, 64, False)]):
        rng = np.random.default_rng(500 + seed)
        rp, col = _rand_graph(600 + seed, n, 20, multi)
        x = rng.standard_normal((n, H, d)).astype(np.float32)
        w = rng.standard_normal((col.size, H)).astype(np.float32)
        want = np.zeros((n, H, d))
        for dst in range(n):
            a, b = rp[dst], rp[dst + 1]
            if b > a:
                want[dst] = (x[col[a:b]].astype(np.float64) * w[a:b, :, None].astype(np.float64)).sum(0)
        got = agg(rp, col, n, H, d, "f32", w, x)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), np.abs(got - want).max()


def pin_aggregate_index_add(agg):
    """The article's normalised scatter-add: two index_add_ scatters (sum of scaled
    values, sum of scores) and numerator / (denominator + eps), in torch fp64."""
    import torch

    n, H, d = 37, 4, 16
    rng = np.random.default_rng(71)
    rp, col = _rand_graph(72, n, 15, True)
    x = rng.standard_normal((n, H, d)).astype(np.float32)
    w = rng.random((col.size, H)).astype(np.float32) + 0.1
    dst = torch.from_numpy(np.repeat(np.arange(n), np.diff(rp)))
    v_scaled = torch.from_numpy(x).double()[torch.from_numpy(col.astype(np.int64))] * torch.from_numpy(w).double()[:, :, None]
    num = torch.zeros(n, H, d, dtype=torch.float64).index_add_(0, dst, v_scaled)
    den = torch.zeros(n, H, 1, dtype=torch.float64).index_add_(0, dst, torch.from_numpy(w).double()[:, :, None])
    want = (num / (den + EPS)).numpy()
    got = agg(rp, col, n, H, d, "f32", w, x, normalize=True, eps=EPS)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)
    got0 = agg(rp, col, n, H, d, "f32", w, x)
    assert np.allclose(got0, num.numpy(), rtol=1e-12, atol=1e-13)


def pin_aggregate_closed_forms(agg):
    rp, col, q, k, v, _ = _graph_and_values(91)
    n, H, d = v.shape
    deg = np.diff(rp)
    ones = np.ones((col.size, H), np.float32)
    sums = np.zeros((n, H, d))
    for i in range(n):
        if deg[i]:
            sums[i] = v[col[rp[i]:rp[i + 1]]].astype(np.float64).sum(0)
    assert np.allclose(agg(rp, col, n, H, d, "f32", ones, v), sums, rtol=1e-13, atol=1e-14)
    want = sums / (deg[:, None, None] + 0.5)
    assert np.allclose(agg(rp, col, n, H, d, "f32", ones, v, normalize=True, eps=0.5), want, rtol=1e-13, atol=1e-14)
    zero = np.zeros_like(ones)
    out = agg(rp, col, n, H, d, "f32", zero, v, normalize=True, eps=1e-6)
    assert np.all(out == 0.0)


AGG_PINS = [pin_aggregate_reference_loop, pin_aggregate_index_add, pin_aggregate_closed_forms]


ALL_PINS = [
    pin_four_node_standard,
    pin_four_node_rtmscore,
    pin_brute_force_standard,
    pin_brute_force_rtmscore,
    pin_permutation_invariance,
    pin_zero_degree_and_weights,
    pin_convex_hull,
    pin_closed_forms,
    pin_clip_bounds,
    pin_library_softmax,
    pin_sixteen_bit_inputs,
]
