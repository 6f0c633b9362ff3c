"""GPU parity of the tensor-core tile path (tcgen05 + TMEM over BSB tiles)."""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, assert_close_stored16, cast_values, device, ensure_built, run_case, upload_graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


def _run(g, H, dtype, plan_kw, seed=7):
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, 64, False, seed=seed)
    plan, O, errs = run_case(g, vals, H, 64, dtype, "standard", plan_kw=plan_kw)
    plan.check()  # no bounded device wait gave up
    return plan, O, vals


def test_tile_small_batched_dense():
    g = graphgen.batched_dense(num_graphs=24, seed=3)
    plan, _, _ = _run(g, 8, "bf16", dict(tile_path=1, tile_density_milli=150, tile_pool_density_milli=0))
    st = plan.stats()
    assert st["tile_path"] == 1 and st["tile_windows"] > 0


def test_full_batched_dense_on_tile_path():
    """The batched dense-ish workload at full size with its windows on the tile path."""
    g, vals, w = graphgen.make_workload("batched_dense", "full")
    plan, _, _ = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant,
                          plan_kw=dict(tile_path=1, tile_density_milli=150, tile_pool_density_milli=0))
    plan.check()
    assert plan.stats()["tile_windows"] > 0.8 * plan.stats()["windows"]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tile_matches_core_path(dtype):
    ensure_built()
    g = graphgen.batched_dense(num_graphs=40, seed=5)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 4, 64, False, seed=9)
    t = {k: v.to(device()) for k, v in cast_values(vals, dtype).items()}
    rp, ci = upload_graph(g)
    tile = g3s.Plan(rp, ci, g.num_nodes, 4, 64, dtype, tile_path=1, tile_density_milli=0, tile_pool_density_milli=0)
    core = g3s.Plan(rp, ci, g.num_nodes, 4, 64, dtype, tile_path=0)
    assert tile.stats()["tile_windows"] == (g.num_nodes + 15) // 16  # every window dense enough
    assert core.stats()["tile_windows"] == 0
    Ot = tile.forward(t["Q"], t["K"], t["V"])
    Oc = core.forward(t["Q"], t["K"], t["V"])
    tile.check()
    want = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, 4, 64, dtype, "standard",
                          *(cast_values(vals, dtype)[k] for k in "QKV"))
    assert_close(Ot, want, dtype, "O tile path")
    assert_close(Oc, want, dtype, "O core path")


def test_tile_mixed_with_core_rows():
    """Some windows dense (tile path), others sparse or holding heavy rows (core path)."""
    a = graphgen.batched_dense(num_graphs=30, seed=11)       # dense windows
    b = graphgen.powerlaw(num_nodes=2003, max_degree=1500, seed=12)  # sparse windows, heavy rows
    off = a.num_nodes
    rp = np.concatenate([a.row_ptr, a.row_ptr[-1] + b.row_ptr[1:]]).astype(np.int32)
    col = np.concatenate([a.col_idx, b.col_idx + off]).astype(np.int32)
    g = graphgen.Graph(rp, col)
    plan, _, _ = _run(g, 2, "bf16", dict(tile_path=1, tile_density_milli=150, tile_pool_density_milli=0, heavy_threshold=60, chunk_edges=25, small_graph_rows=0))
    st = plan.stats()
    assert 0 < st["tile_windows"] < st["windows"] and st["chunks"] > 0


def test_tile_full_windows():
    """Windows of 16 rows with up to 128 unique sources: 16 tiles, the most a
    tile-path window takes (every MMA row a column of the window, eight
    16-column steps of the second product)."""
    rng = np.random.default_rng(13)
    n = 16 * 24 + 5
    cols = []
    deg = np.zeros(n, np.int64)
    for i in range(n):
        w = i // 16
        pool = (np.arange(128) * 3 + w * 17) % n  # 128 distinct sources per window
        s = np.sort(rng.choice(pool, size=rng.integers(40, 100), replace=False))
        cols.append(s)
        deg[i] = s.size
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    g = graphgen.Graph(rp, np.concatenate(cols).astype(np.int32))
    plan, _, _ = _run(g, 2, "f16", dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0, heavy_threshold=512))
    st = plan.stats()
    assert st["tile_windows"] == (n + 15) // 16
    assert st["tiles"] >= 15 * st["tile_windows"]


def test_tile_windows_over_the_limit_stay_on_core():
    """With split windows off, a window with more than 16 tiles (over 128
    unique sources) goes to the CUDA-core kernel; the others of the same graph
    take the tile path."""
    rng = np.random.default_rng(14)
    n = 16 * 6
    cols, deg = [], np.zeros(n, np.int64)
    for i in range(n):
        span = 200 if i < 16 else 60  # window 0 draws from 200 sources: over 16 tiles
        s = np.sort(rng.choice(span, size=rng.integers(30, 50), replace=False))
        cols.append(s)
        deg[i] = s.size
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    nn = 200
    rp = np.concatenate([rp, np.full(nn - n, rp[-1], np.int32)])
    g = graphgen.Graph(rp, np.concatenate(cols).astype(np.int32))
    vals = graphgen.make_values(nn, g.num_edges, 2, 64, False, seed=15)
    plan, _, _ = run_case(g, vals, 2, 64, "bf16", "standard",
                          plan_kw=dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0,
                                       tile_split_density_milli=0))
    plan.check()
    flags = plan.export("win_flags")
    assert not (flags[0] & 2) and all(flags[1:6] & 2)


def test_tile_wide_logit_range():
    """Windows of 16 tiles whose later columns carry much larger logits
    (spread over tens of units): the row max over all of a window's columns
    is taken before any P is formed, so no term overflows and the small ones
    vanish as they should."""
    rng = np.random.default_rng(29)
    n = 16 * 8
    cols, deg = [], np.zeros(n, np.int64)
    for i in range(n):
        s = np.sort(rng.choice(128, size=rng.integers(60, 110), replace=False))  # sources 0..127, sorted
        cols.append(s)
        deg[i] = s.size
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    nn = 256
    rp = np.concatenate([rp, np.full(nn - n, rp[-1], np.int32)])  # nodes 128..255: no in-edges
    g = graphgen.Graph(rp, np.concatenate(cols).astype(np.int32))
    vals = graphgen.make_values(nn, g.num_edges, 2, 64, False, seed=30)
    ramp = np.linspace(0.2, 6.0, nn, dtype=np.float32)[:, None, None]  # logits grow with the column id
    vals["K"] = np.abs(vals["K"] * ramp)
    vals["Q"] = np.abs(vals["Q"]) * 2.0
    plan, _, _ = run_case(g, vals, 2, 64, "bf16", "standard",
                          plan_kw=dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0, heavy_threshold=512))
    plan.check()
    assert plan.stats()["tile_windows"] == 8


def test_tile_multigraph_windows_stay_on_core():
    g = graphgen.random_csr(200, 30, seed=17, multigraph=True)
    plan, _, _ = _run(g, 2, "bf16", dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0))
    flags = plan.export("win_flags")
    assert np.any(flags & 1)  # the multigraph has windows with repeated edges
    assert not np.any(((flags & 1) != 0) & ((flags & 2) != 0))  # none of them takes the tile path


def test_tile_sixteen_bit_output():
    g = graphgen.batched_dense(num_graphs=16, seed=19)
    plan, O, _ = _run(g, 8, "bf16", dict(tile_path=1, out_dtype="bf16", tile_density_milli=150, tile_pool_density_milli=0))
    assert O.dtype == torch.bfloat16 and plan.stats()["tile_windows"] > 0


def test_tile_rows_with_no_edges():
    rng = np.random.default_rng(23)
    n = 64
    deg = rng.integers(5, 20, n)
    deg[[3, 17, 18, 40]] = 0
    cols = [np.sort(rng.choice(n, size=d, replace=False)) for d in deg]
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    g = graphgen.Graph(rp, np.concatenate(cols).astype(np.int32))
    plan, O, _ = _run(g, 1, "bf16", dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0))
    assert plan.stats()["tile_windows"] == 4
    assert torch.count_nonzero(O[[3, 17, 18, 40]]).item() == 0


@pytest.mark.parametrize("H", [1, 8])
def test_tile_mixed_full_size_persistent_core_rows(H):
    """Full-size batched graphs with p = 0.5 and a per-window density cutoff
    of 0.4: about 60% of the windows on tiles and the rest left to the
    CUDA-core kernel's window list (both kernels in one forward), with more
    of those rows than resident warps (its persistent loop).  H = 1 also
    takes the short-row pack flavour beside the tile windows.  Sampled rows
    and both ends are checked."""
    g = graphgen.batched_dense(num_graphs=1024, p=0.5, seed=1003)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, 64, False, seed=2003)
    rows = np.unique(np.concatenate([np.random.default_rng(17).choice(g.num_nodes, 4000, replace=False),
                                     np.arange(16), g.num_nodes - 1 - np.arange(16)]))
    plan, _, _ = run_case(g, vals, H, 64, "bf16", "standard", rows=rows,
                          plan_kw=dict(pack_rows=1 if H == 1 else -1, tile_density_milli=400,
                                       tile_pool_density_milli=0))
    plan.check()
    st = plan.stats()
    core_rows = 16 * (st["windows"] - st["tile_windows"])
    assert 0 < st["tile_windows"] < st["windows"] and core_rows > 152 * 8 * 3


# ---------------------------------------------------------------------------
# the device planner's tile-path selection, bit-exact with the tile path on
# ---------------------------------------------------------------------------
def _split_graph():
    from test_planner_oracle import _split_graph as make  # the reference planner's split-window pin graph
    return make()


def _mixed_graph():
    a = graphgen.batched_dense(num_graphs=30, seed=11)
    b = graphgen.powerlaw(num_nodes=2003, max_degree=1500, seed=12)
    rp = np.concatenate([a.row_ptr, a.row_ptr[-1] + b.row_ptr[1:]]).astype(np.int32)
    col = np.concatenate([a.col_idx, b.col_idx + a.num_nodes]).astype(np.int32)
    return graphgen.Graph(rp, col)


def _selection_cases():
    """(name, graph, heads, plan options, whether windows take the tile path)"""
    dense_full = lambda: graphgen.make_workload("batched_dense", "full")[0]  # noqa: E731
    complete_small = lambda: graphgen.make_workload("batched_complete", "small")[0]  # noqa: E731
    per_window = dict(tile_density_milli=150, tile_pool_density_milli=0)
    yield "batched_dense_full_default", dense_full, 8, {}, True  # pooled density 0.24 >= 0.18
    yield "batched_dense_full_pool_300", dense_full, 8, dict(tile_pool_density_milli=300), False
    yield "batched_dense_full_per_window", dense_full, 8, per_window, True
    yield "batched_dense_full_per_window_global_bitmap", dense_full, 8, dict(per_window, bsb_smem_edges=64), True
    yield "batched_complete_small", complete_small, 8, {}, True
    yield "batched_complete_small_global_bitmap", complete_small, 8, dict(bsb_smem_edges=100), True
    yield "mixed_heavy", _mixed_graph, 2, dict(per_window, heavy_threshold=60, chunk_edges=25, small_graph_rows=0), True
    yield "mixed_heavy_pooled_out", _mixed_graph, 2, dict(tile_pool_density_milli=500, heavy_threshold=60,
                                                         chunk_edges=25, small_graph_rows=0), False
    yield "mixed_heavy_global_bitmap", _mixed_graph, 2, dict(per_window, heavy_threshold=60, chunk_edges=25, small_graph_rows=0,
                                                            bsb_smem_edges=48), True
    yield "mixed_max_tiles", _mixed_graph, 2, dict(tile_density_milli=0, tile_pool_density_milli=0,
                                                   tile_max_tiles=5), True
    # a floor of 0.25 keeps the pin graph's sparse wide windows on CUDA cores
    split_kw = dict(heavy_threshold=100, chunk_edges=64, small_graph_rows=0, tile_split_density_milli=250)
    yield "split_mixed", _split_graph, 2, split_kw, True
    yield "split_default_floor", _split_graph, 2, dict(heavy_threshold=100, chunk_edges=64, small_graph_rows=0), True
    yield "split_mixed_edge", _split_graph, 2, dict(split_kw, tile_split_parallel=1), True
    yield "split_mixed_global_bitmap", _split_graph, 2, dict(split_kw, bsb_smem_edges=256), True
    yield "split_mixed_edge_global_bitmap", _split_graph, 2, dict(split_kw, bsb_smem_edges=256, tile_split_parallel=1), \
        True
    yield "split_mixed_dense_only", _split_graph, 2, dict(split_kw, tile_split_density_milli=600), True
    yield "split_off", _split_graph, 2, dict(split_kw, tile_split_density_milli=0), True
    yield "clustered_small", lambda: graphgen.make_workload("clustered_heavy", "small")[0], 8, \
        dict(heavy_threshold=150), True


@pytest.mark.parametrize("name,make,H,kw,tiled", list(_selection_cases()), ids=[c[0] for c in _selection_cases()])
def test_tile_selection_bit_exact(name, make, H, kw, tiled):
    """With the tile path on, the device planner's BSB arrays, window flags
    (bit 1 = tile path), the tile-path window list and the list of windows
    left to the CUDA-core kernel equal the reference planner's, through both
    window-compaction kernels (shared-memory sort and global bitmap)."""
    from oracle import planner as ref_planner
    g = make()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, 64, "bf16", tile_path=1, **kw)
    st = plan.stats()
    opts = g3s.make_options(tile_path=1, **kw)
    b = ref_planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    sel = ref_planner.tile_selection(g.row_ptr, b, True, heavy_threshold=st["heavy_threshold"],
                                     max_tiles=opts.tile_max_tiles, density_milli=opts.tile_density_milli,
                                     pool_milli=opts.tile_pool_density_milli,
                                     split_milli=opts.tile_split_density_milli)
    hc = ref_planner.heavy_chunks(g.row_ptr, st["heavy_threshold"], st["chunk_edges"])
    n_chunks = hc["chunks"].shape[0]
    ref = dict(b, **sel)
    for arr in ("win_tile_ptr", "tile_cols", "tile_bits", "win_nnz", "win_flags", "tile_windows", "core_windows"):
        got = plan.export(arr)
        want = ref[arr]
        assert got.shape == want.shape and np.array_equal(got, want.astype(got.dtype)), arr
    tw, sw = sel["tile_windows"], sel["split_windows"]
    assert st["tile_windows"] == tw.size + sw.size and st["split_windows"] == sw.size
    assert st["tile_window_nnz"] == int(b["win_nnz"][tw].sum() + b["win_nnz"][sw].sum())
    edge = opts.tile_split_parallel == 1
    want_items = ref_planner.tile_items(g.row_ptr, b, tw, sw, n_chunks, edge)
    got_items = plan.export("tile_items")
    assert st["tile_items"] == want_items.shape[0]
    assert got_items.shape == want_items.shape and np.array_equal(got_items, want_items), "tile_items"
    if sw.size:
        ml = ref_planner.merge_list(g.row_ptr, b, sel["win_flags"], st["heavy_threshold"], hc["heavy_chunk_ptr"],
                                    n_chunks, edge)
        assert st["merge_rows"] == ml["merge_rows"].size
        assert np.array_equal(plan.export("merge_rows"), ml["merge_rows"]), "merge_rows"
        assert np.array_equal(plan.export("merge_ranges"), ml["merge_ranges"]), "merge_ranges"
    if name.startswith("split_mixed"):
        assert sw.size > 0 and tw.size > 0 and st["chunks"] > 0
    if "bsb_smem_edges" in kw:
        assert st["large_windows"] > 0
    assert (st["tile_windows"] > 0) == tiled
    if name.startswith("mixed") and tiled:
        assert 0 < st["tile_windows"] < st["windows"]


# ---------------------------------------------------------------------------
# split windows: windows wider than 128 columns cut into 128-column slices
# whose partial softmax states are merged per row
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("parallel", [0, 1], ids=["node", "edge"])
@pytest.mark.parametrize("dtype,H", [("bf16", 2), ("f16", 4), ("bf16", 8)])
def test_split_windows_parity(dtype, H, parallel):
    """Split windows (heavy rows, light rows and empty rows in them), pairs,
    CUDA-core windows and heavy-row chunks outside the split windows in one
    plan, every row against the oracle; node-parallel (chains) and
    edge-parallel (slices merged)."""
    g = _split_graph()
    plan, _, _ = _run(g, H, dtype, dict(tile_path=1, heavy_threshold=100, chunk_edges=64, small_graph_rows=0,
                                        tile_split_parallel=parallel, tile_split_density_milli=250))
    st = plan.stats()
    assert st["split_windows"] > 0 and st["tile_windows"] > st["split_windows"]
    assert st["windows"] > st["tile_windows"] and st["chunks"] > 0
    # every heavy row of this graph sits in a split window: merged from its
    # slices edge-parallel, final in the tile kernel node-parallel
    assert (st["merge_rows"] > 0) == (parallel == 1)


def test_split_windows_off():
    g = _split_graph()
    plan, _, _ = _run(g, 2, "bf16", dict(tile_path=1, heavy_threshold=100, chunk_edges=64,
                                         tile_split_density_milli=0))
    assert plan.stats()["split_windows"] == 0


@pytest.mark.parametrize("parallel", [0, 1], ids=["node", "edge"])
def test_split_windows_sixteen_bit_output(parallel):
    g = _split_graph()
    plan, O, _ = _run(g, 2, "bf16", dict(tile_path=1, heavy_threshold=100, chunk_edges=64, out_dtype="bf16",
                                         tile_split_parallel=parallel))
    assert O.dtype == torch.bfloat16 and plan.stats()["split_windows"] > 0


@pytest.mark.parametrize("parallel", [0, 1], ids=["node", "edge"])
def test_clustered_heavy_small_workload(parallel):
    """Every window split (two slices of 16 and 8 tiles), every heavy row
    inside a split window (its chunks skipped), a ragged last window, empty
    rows."""
    g, vals, w = graphgen.make_workload("clustered_heavy", "small")
    plan, _, _ = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant,
                          plan_kw=dict(heavy_threshold=150, tile_split_parallel=parallel))
    plan.check()
    st = plan.stats()
    assert st["split_windows"] == st["windows"] and st["chunks"] > 0 and g.num_nodes % 16
    assert st["merge_rows"] == (g.num_nodes if parallel else 0)
    assert np.any(g.degrees() == 0)


def test_chain_rescale_across_slices():
    """Node-parallel chains whose later slices carry much larger logits than
    the first (the reference max moves, O and the row sums are rescaled in
    TMEM), and rows whose first slices are empty."""
    rng = np.random.default_rng(31)
    n = 16 * 8
    cols, deg = [], np.zeros(n, np.int64)
    for i in range(n):
        lo = 0 if i % 3 else 256  # every third row has nothing in the first two slices
        s = np.sort(rng.choice(np.arange(lo, 512), size=160, replace=False))
        cols.append(s)
        deg[i] = s.size
    nn = 512
    rp = np.zeros(nn + 1, np.int32)
    rp[1:n + 1] = np.cumsum(deg)
    rp[n + 1:] = rp[n]
    g = graphgen.Graph(rp, np.concatenate(cols).astype(np.int32))
    vals = graphgen.make_values(nn, g.num_edges, 2, 64, False, seed=32)
    vals["K"][256:] *= 6.0  # logits of the last two slices' columns far above the first ones'
    for parallel in (0, 1):
        plan, _, _ = run_case(g, vals, 2, 64, "bf16", "standard",
                              plan_kw=dict(tile_path=1, tile_split_parallel=parallel))
        plan.check()
        st = plan.stats()
        assert st["split_windows"] == 8 and st["split_items"] == 8 * 4


def test_clustered_heavy_full_sampled_rows():
    """The full clustered workload in the bench's launch configuration (default
    plan), on every row of four windows and 2000 random rows."""
    g, vals, w = graphgen.make_workload("clustered_heavy", "full")
    W = (g.num_nodes + 15) // 16
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(16 * 500, 16 * 501), np.arange(16 * (W - 2), g.num_nodes),
                                     rng.choice(g.num_nodes, 2000, replace=False)]))
    plan, _, _ = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant, rows=rows)
    plan.check()
    st = plan.stats()
    assert st["split_windows"] > 0.97 * W and st["split_items"] > 16 * st["split_windows"]


def test_split_plan_aggregate():
    """g3s_aggregate on a plan with split windows takes every row through the
    CUDA-core kernel and the heavy-row chunks (the split windows are the
    forward's alone)."""
    g = _split_graph()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 2, 64, "bf16", tile_path=1, heavy_threshold=100, chunk_edges=64)
    assert plan.stats()["split_windows"] > 0
    rng = np.random.default_rng(5)
    wt = torch.from_numpy(rng.random((g.num_edges, 2), dtype=np.float32) + 0.1).to(torch.bfloat16)
    xt = torch.from_numpy(rng.standard_normal((g.num_nodes, 2, 64), dtype=np.float32)).to(torch.bfloat16)
    O = plan.aggregate(wt.to(device()), xt.to(device()), normalize=True, eps=1e-6)
    torch.cuda.synchronize()
    want = oracle.aggregate(g.row_ptr, g.col_idx, g.num_nodes, 2, 64, "bf16", wt, xt, normalize=True, eps=1e-6)
    assert_close(O, want, "bf16", "O (aggregate)")


def _wide_window_graph(nnz_first: int, dup: bool, seed: int):
    """Two 16-row windows over 160 source columns (20 tiles): the first holds
    nnz_first entries (a row repeats a source when dup), the second is the
    same pattern over columns shifted by 8; then 160 empty rows."""
    rng = np.random.default_rng(seed)
    n = 192
    rows = [[] for _ in range(n)]
    for w in (0, 1):
        cols = np.arange(160) + 8 * w  # every column used at least once
        per = [nnz_first // 16 + (1 if r < nnz_first % 16 else 0) for r in range(16)]
        pool = list(cols)
        rng.shuffle(pool)
        k = 0
        for r in range(16):
            take = [pool[(k + j) % 160] for j in range(per[r])]
            k += per[r]
            rows[16 * w + r] = sorted(set(take))
        if dup and w == 0:
            rows[3] = sorted(rows[3] + [rows[3][0]])
    deg = np.array([len(x) for x in rows])
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    col = np.concatenate([np.asarray(x, np.int64) for x in rows if x]).astype(np.int32)
    return graphgen.Graph(rp, col)


@pytest.mark.parametrize("nnz,dup,split", [(640, False, True), (639, False, False), (800, True, False)],
                         ids=["at_threshold", "one_below", "repeated_pair"])
def test_split_density_boundary_and_repeated_pairs(nnz, dup, split):
    """A 20-tile window whose density is exactly 0.25 (640 entries) splits,
    one entry fewer does not, and a dense window holding a repeated (row,
    source) pair never does (it runs on CUDA cores); the device planner
    matches the reference planner and O matches the oracle."""
    from oracle import planner as ref_planner
    g = _wide_window_graph(nnz, dup, seed=41)
    b = ref_planner.bsb(g.row_ptr, g.col_idx, g.num_nodes)
    assert int(np.diff(b["win_tile_ptr"])[0]) == 20 and int(b["win_nnz"][0]) == nnz + (1 if dup else 0)
    plan, _, _ = _run(g, 2, "bf16", dict(tile_path=1, heavy_threshold=512, tile_split_density_milli=250))
    flags = plan.export("win_flags")
    assert bool(flags[0] & 8) == split and bool(flags[0] & 1) == dup
    sel = ref_planner.tile_selection(g.row_ptr, b, True, heavy_threshold=512, max_tiles=16, density_milli=100,
                                     pool_milli=180, split_milli=250)
    assert np.array_equal(flags, sel["win_flags"])
