"""GPU parity of the short-row packs of the fused kernel (plan option
pack_rows): where a node row is at most 256 bytes, a warp takes G = 32 /
row_vecs consecutive rows together, one per lane group, when each has at
most min(4 G, 2 * 32 / G) entries (and no more than the heavy-row
threshold); packs holding a longer row fall back to one row per warp.  The
kernel with packs is a second flavour, taken by default when at least a
quarter of the rows are short.

Checked against the fp64 oracle with packing on and off, for every row
width that packs, on degree mixes around the pack limit, with empty rows, a
ragged last pack, heavy rows among short ones, a heavy-row threshold below
the pack limit, tile-path windows beside packed rows, and both launch forms
(one item per warp for small graphs, the persistent loop for large ones).
"""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, device, ensure_built, run_case, upload_graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


ELT = {"f32": 4, "f16": 2, "bf16": 2}


def pack_limit(H, d, dtype, heavy_threshold=512):
    rv = H * d * ELT[dtype] // 16
    G = 32 // rv
    return min(4 * G, 2 * (32 // G), heavy_threshold), G


def graph_with_degrees(degs, num_nodes, seed):
    """Simple graph whose row i has degs[i] distinct sources (ascending)."""
    rng = np.random.default_rng(seed)
    cols = [np.sort(rng.choice(num_nodes, int(k), replace=False)) for k in degs]
    row_ptr = np.zeros(len(degs) + 1, np.int64)
    row_ptr[1:] = np.cumsum(degs)
    col = np.concatenate(cols) if len(cols) else np.zeros(0, np.int64)
    return graphgen.Graph(row_ptr.astype(np.int32), col.astype(np.int32))


def short_mix(n, limit, seed, long_frac=0.03, long_max=700):
    """Degrees 0..limit+1 (most rows packable), a few long ones up to long_max."""
    rng = np.random.default_rng(seed)
    degs = rng.integers(0, limit + 2, n)
    longs = rng.random(n) < long_frac
    degs[longs] = rng.integers(limit + 2, long_max, longs.sum())
    degs[:8] = 0                       # a pack of empty rows
    degs[8:16] = limit                 # packs exactly at the limit
    degs[16:24] = [limit + 1] + [1] * 7  # one row just over it
    return np.minimum(degs, n)


# (dtype, heads, head_dim): node rows of 32 to 256 bytes (G = 16 .. 2)
SHAPES = [("bf16", 4, 32), ("f16", 1, 64), ("bf16", 1, 64), ("f16", 1, 32), ("bf16", 1, 16), ("f32", 1, 16),
          ("f32", 2, 32), ("f32", 1, 32), ("f16", 2, 16), ("bf16", 8, 16)]


@pytest.mark.parametrize("dtype,H,d", SHAPES, ids=["%s-%dx%d" % s for s in SHAPES])
@pytest.mark.parametrize("pack", [1, 0])
def test_pack_matches_oracle(dtype, H, d, pack):
    limit, G = pack_limit(H, d, dtype)
    n = 997  # not a multiple of any pack size
    g = graph_with_degrees(short_mix(n, limit, seed=1), n, seed=2)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, d, False, seed=3)
    plan, _, _ = run_case(g, vals, H, d, dtype, "standard",
                          plan_kw=dict(heavy_threshold=300, chunk_edges=37, small_graph_rows=0, pack_rows=pack))
    st = plan.stats()
    assert st["chunks"] > 0 and st["pack_rows"] == pack


@pytest.mark.parametrize("dtype,H,d", [("f16", 1, 64), ("bf16", 4, 32), ("f32", 1, 16)])
def test_pack_heavy_threshold_below_limit(dtype, H, d):
    """A heavy-row threshold under the pack limit: rows above it go to chunks,
    never into a pack."""
    n = 515
    rng = np.random.default_rng(4)
    g = graph_with_degrees(rng.integers(0, 12, n), n, seed=5)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, d, False, seed=6)
    plan, _, _ = run_case(g, vals, H, d, dtype, "standard",
                          plan_kw=dict(heavy_threshold=3, chunk_edges=2, small_graph_rows=0, pack_rows=1))
    st = plan.stats()
    assert st["heavy_rows"] > 0 and st["pack_rows"] == 1 and st["pack_limit"] == 3


@pytest.mark.parametrize("out", ["f32", "same"])
def test_pack_stored_16bit_output(out):
    n = 1200
    limit, _ = pack_limit(1, 64, "f16")
    g = graph_with_degrees(short_mix(n, limit, seed=7), n, seed=8)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 1, 64, False, seed=9)
    plan, _, _ = run_case(g, vals, 1, 64, "f16", "standard",
                          plan_kw=dict(out_dtype="f16" if out == "same" else "f32", pack_rows=1))
    assert plan.stats()["pack_rows"] == 1


def test_pack_beside_tile_windows():
    """Tile-path windows (whole 16-row windows) next to packed rows."""
    g = graphgen.batched_dense(num_graphs=40, seed=10)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 1, 64, False, seed=11)
    plan, _, _ = run_case(g, vals, 1, 64, "bf16", "standard",
                          plan_kw=dict(tile_path=1, tile_density_milli=300, tile_pool_density_milli=0, pack_rows=1))
    st = plan.stats()
    assert 0 < st["tile_windows"] < st["windows"] and st["pack_rows"] == 1


def test_pack_auto_choice_and_counts():
    """The planner counts rows with at most pack_limit entries; the default
    takes packs when they are at least a quarter of the rows."""
    rp_cases = [(graphgen.powerlaw(num_nodes=20_000, seed=21), 1, 64, "f16", 1),
                (graphgen.lognormal_local(num_nodes=20_000, radius=512, seed=22), 4, 32, "bf16", 0),
                (graphgen.tiny_poisson(seed=23), 8, 32, "f32", 0)]  # 1 KB rows: no packs
    for g, H, d, dtype, want in rp_cases:
        rp, ci = upload_graph(g)
        st = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype).stats()
        rv = H * d * ELT[dtype] // 16
        limit = pack_limit(H, d, dtype)[0] if rv <= 16 else 0
        deg = np.diff(g.row_ptr)
        assert st["pack_limit"] == limit
        assert st["short_rows"] == (int((deg <= limit).sum()) if limit else 0)
        assert st["pack_rows"] == want
        assert g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, pack_rows=0).stats()["pack_rows"] == 0
        assert g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, pack_rows=1).stats()["pack_rows"] == (1 if limit else 0)


def test_pack_persistent_launch():
    """Enough packs that the kernel runs its persistent loop (more items than
    resident warps); sampled rows and both ends checked."""
    g = graphgen.powerlaw(num_nodes=120_000, seed=12)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 1, 64, False, seed=13)
    rows = np.unique(np.concatenate([np.random.default_rng(14).choice(g.num_nodes, 3000, replace=False),
                                     np.arange(8), g.num_nodes - 1 - np.arange(8)]))
    plan, _, _ = run_case(g, vals, 1, 64, "f16", "standard", rows=rows)
    assert plan.stats()["pack_rows"] == 1  # the default takes packs here


def test_pack_and_no_pack_agree():
    """The same plan inputs with and without packs: both within the oracle's
    tolerance, and within rounding of each other."""
    n = 3001
    limit, _ = pack_limit(4, 32, "bf16")
    g = graph_with_degrees(short_mix(n, limit, seed=15), n, seed=16)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 4, 32, False, seed=17)
    _, O1, _ = run_case(g, vals, 4, 32, "bf16", "standard", plan_kw=dict(pack_rows=1))
    _, O0, _ = run_case(g, vals, 4, 32, "bf16", "standard", plan_kw=dict(pack_rows=0))
    assert torch.allclose(O1, O0, rtol=0, atol=1e-5)


@pytest.mark.parametrize("normalize", [False, True])
@pytest.mark.parametrize("pack", [1, 0])
def test_pack_aggregate(normalize, pack):
    """The weighted aggregation takes the same packs."""
    H, d, dtype = 2, 16, "bf16"
    limit, _ = pack_limit(H, d, dtype)
    n = 777
    g = graph_with_degrees(short_mix(n, limit, seed=18), n, seed=19)
    rng = np.random.default_rng(20)
    x = rng.standard_normal((g.num_nodes, H, d)).astype(np.float32)
    w = np.abs(rng.standard_normal((g.num_edges, H)).astype(np.float32)) + 0.05
    xt, wt = graphgen.to_dtype(x, dtype), graphgen.to_dtype(w, dtype)
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, pack_rows=pack)
    assert plan.stats()["pack_rows"] == pack
    O = plan.aggregate(wt.to(device()), xt.to(device()), normalize=normalize)
    torch.cuda.synchronize()
    want = oracle.aggregate(g.row_ptr, g.col_idx, g.num_nodes, H, d, dtype, wt, xt, normalize=normalize)
    assert_close(O, want, dtype, "O (aggregate)")
