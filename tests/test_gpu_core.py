"""GPU parity of the CUDA-core fused path and the device planner, through the
C ABI, against the fp64 oracle and the numpy reference planner."""
import ctypes

import numpy as np
import pytest
import torch

import graphgen
import oracle
from oracle import planner as ref_planner
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, cast_values, device, ensure_built, run_case, upload_graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(graphgen.WORKLOADS))
def test_small_workload(name):
    g, vals, w = graphgen.make_workload(name, "small")
    run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant)


@pytest.mark.parametrize("name", ["tiny_poisson", "rtmscore_batch64", "batched_dense", "powerlaw", "batched_complete"])
def test_full_workload_all_rows(name):
    g, vals, w = graphgen.make_workload(name, "full")
    run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant)


def test_full_lognormal_all_rows():
    """The large HBM-bound workload at full size (2M rows, ~100M edges), in
    the launch configuration the benchmark times, checked on every row
    against the oracle (heavy rows split into chunks included)."""
    g, vals, w = graphgen.make_workload("lognormal_local", "full")
    plan, _, errs = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant)
    assert plan.stats()["chunks"] > 0


@pytest.mark.parametrize("name", ["batched_dense", "powerlaw", "lognormal_local"])
def test_sixteen_bit_output(name):
    """O stored in the 16-bit input type (plan option out_dtype)."""
    g, vals, w = graphgen.make_workload(name, "small")
    plan, O, _ = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant,
                          plan_kw=dict(out_dtype=w.dtype, heavy_threshold=64, chunk_edges=40, small_graph_rows=0))
    assert O.dtype == {"bf16": torch.bfloat16, "f16": torch.float16}[w.dtype]


def test_sixteen_bit_rtmscore_eout():
    g = graphgen.rtmscore_batch(num_graphs=3, min_nodes=30, max_nodes=60, seed=16)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 8, 16, True, seed=17)
    for dt in ("bf16", "f16"):
        run_case(g, vals, 8, 16, dt, "rtmscore", plan_kw=dict(out_dtype=dt, heavy_threshold=8, chunk_edges=5, small_graph_rows=0))
        run_case(g, vals, 8, 16, dt, "rtmscore", plan_kw=dict(heavy_threshold=8, chunk_edges=5, small_graph_rows=0))


# ---------------------------------------------------------------------------
# heavy-row split + merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,variant", [("f32", "standard"), ("bf16", "standard"), ("f32", "rtmscore"),
                                           ("f16", "rtmscore")])
def test_heavy_split_matches_oracle(dtype, variant):
    g = graphgen.powerlaw(num_nodes=3000, max_degree=2000, seed=5)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 2, 32, variant == "rtmscore", seed=6)
    plan, O, _ = run_case(g, vals, 2, 32, dtype, variant, plan_kw=dict(heavy_threshold=20, chunk_edges=7, small_graph_rows=0))
    st = plan.stats()
    assert st["heavy_rows"] > 50 and st["chunks"] > st["heavy_rows"]


# ---------------------------------------------------------------------------
# shapes: every lane mapping (groups per warp, vectors per lane)
# ---------------------------------------------------------------------------
SHAPES = [("f32", 1, 16), ("f32", 2, 32), ("f32", 8, 32), ("f32", 4, 128), ("f32", 8, 128),
          ("bf16", 1, 16), ("bf16", 1, 64), ("bf16", 4, 32), ("bf16", 8, 64), ("bf16", 16, 128),
          ("f16", 2, 16), ("f16", 1, 128), ("f16", 8, 32)]


@pytest.mark.parametrize("dtype,H,d", SHAPES, ids=["%s-%dx%d" % s for s in SHAPES])
@pytest.mark.parametrize("variant", ["standard", "rtmscore"])
def test_shapes(dtype, H, d, variant):
    g = graphgen.random_csr(133, 45, seed=H * 1000 + d, zero_frac=0.15)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, d, variant == "rtmscore", seed=d + H)
    run_case(g, vals, H, d, dtype, variant, plan_kw=dict(heavy_threshold=30, chunk_edges=9, small_graph_rows=0))


# ---------------------------------------------------------------------------
# the RTMScore variant's readings
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("clamp", [True, False])
def test_rtmscore_clamp_readings(clamp):
    g = graphgen.rtmscore_batch(num_graphs=4, min_nodes=40, max_nodes=80, seed=12)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 8, 16, True, seed=13)
    vals["Q"] *= 6.0  # drive q*k/sqrt(d) and the logits into the clip range
    vals["K"] *= 6.0
    run_case(g, vals, 8, 16, "f32", "rtmscore", oracle_kw=dict(elementwise_clamp=clamp))


def test_rtmscore_without_eout():
    g = graphgen.rtmscore_batch(num_graphs=2, min_nodes=30, max_nodes=50, seed=14)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 8, 16, True, seed=15)
    run_case(g, vals, 8, 16, "f32", "rtmscore", check_eout=False)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
def test_no_edges_gives_zero():
    g = graphgen.Graph(np.zeros(37, np.int32), np.zeros(0, np.int32))
    vals = graphgen.make_values(36, 0, 2, 32, False, seed=1)
    plan, O, _ = run_case(g, vals, 2, 32, "bf16", "standard")
    assert torch.count_nonzero(O).item() == 0


def test_single_node_self_loop():
    g = graphgen.Graph(np.array([0, 1], np.int32), np.array([0], np.int32))
    vals = graphgen.make_values(1, 1, 4, 32, True, seed=2)
    run_case(g, vals, 4, 32, "f32", "standard")
    run_case(g, vals, 4, 32, "f32", "rtmscore")


@pytest.mark.parametrize("multigraph,sorted_rows", [(True, True), (False, False), (True, False)])
def test_multigraph_and_unsorted(multigraph, sorted_rows):
    g = graphgen.random_csr(211, 60, seed=21, zero_frac=0.1, multigraph=multigraph, sorted_rows=sorted_rows)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 4, 32, False, seed=22)
    run_case(g, vals, 4, 32, "bf16", "standard", plan_kw=dict(heavy_threshold=40, chunk_edges=16, small_graph_rows=0))


def test_deterministic_and_edge_order_invariant():
    ensure_built()
    g = graphgen.powerlaw(num_nodes=4000, max_degree=3000, seed=31)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 1, 64, False, seed=32)
    t = cast_values(vals, "f16")
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 1, 64, "f16")
    Q, K, V = (t[k].to(dev) for k in "QKV")
    O1 = plan.forward(Q, K, V).clone()
    O2 = plan.forward(Q, K, V)
    assert torch.equal(O1, O2)
    # permute the edges inside every row: same attention up to rounding
    rng = np.random.default_rng(3)
    col = g.col_idx.copy()
    for i in range(g.num_nodes):
        a, b = g.row_ptr[i], g.row_ptr[i + 1]
        col[a:b] = rng.permutation(col[a:b])
    rp2, ci2 = upload_graph(graphgen.Graph(g.row_ptr, col))
    plan2 = g3s.Plan(rp2, ci2, g.num_nodes, 1, 64, "f16")
    O3 = plan2.forward(Q, K, V)
    assert_close(O3, O1.double().cpu().numpy(), "f16", "O (permuted edges)")


def test_forward_host_matches_forward():
    ensure_built()
    g, vals, w = graphgen.make_workload("rtmscore_batch64", "small")
    t = cast_values(vals, w.dtype)
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant)
    O, Eout = plan.forward(*(t[k].to(dev) for k in "QKV"), t["E"].to(dev), want_eout=True)
    pin = {k: v.pin_memory() for k, v in t.items()}
    Oh = torch.empty_like(pin["Q"]).pin_memory()
    Eoh = torch.empty_like(pin["E"]).pin_memory()
    plan.forward_host(pin["Q"], pin["K"], pin["V"], Oh, pin["E"], Eoh)
    torch.cuda.synchronize()
    assert torch.equal(Oh, O.cpu()) and torch.equal(Eoh, Eout.cpu())


# ---------------------------------------------------------------------------
# device planner, bit-exact against the reference planner
# ---------------------------------------------------------------------------
def _planner_graphs():
    yield "tiny", graphgen.tiny_poisson(), {}
    yield "dense", graphgen.batched_dense(num_graphs=40, seed=3), {}
    yield "powerlaw", graphgen.powerlaw(num_nodes=20000, seed=4), {}
    yield "powerlaw_large_windows", graphgen.powerlaw(num_nodes=20000, seed=4), dict(bsb_smem_edges=64)
    yield "multigraph", graphgen.random_csr(300, 90, seed=5, multigraph=True, sorted_rows=False), dict(bsb_smem_edges=200)
    yield "lognormal", graphgen.lognormal_local(num_nodes=30000, radius=2048, seed=6), {}
    yield "ragged", graphgen.random_csr(17, 9, seed=7, zero_frac=0.3), dict(bsb_smem_edges=5)


@pytest.mark.parametrize("name,g,kw", list(_planner_graphs()), ids=[n for n, _, _ in _planner_graphs()])
def test_planner_bit_exact(name, g, kw):
    ensure_built()
    rp, ci = upload_graph(g)
    opts = dict(bsb=1, heavy_threshold=64, chunk_edges=32, small_graph_rows=0, bucket_bounds=(4, 16, 128), degree_buckets=1)
    opts.update(kw)
    plan = g3s.Plan(rp, ci, g.num_nodes, 2, 32, "bf16", **opts)
    ref = ref_planner.full_plan(g.row_ptr, g.col_idx, g.num_nodes, bounds=(4, 16, 128), heavy_threshold=64,
                                chunk_edges=32, with_bsb=True, tile_enabled=False)
    for name_ in ("bucket_ptr", "bucket_rows", "heavy_rows", "heavy_chunk_ptr", "chunks", "win_tile_ptr",
                  "tile_cols", "tile_bits", "win_nnz", "win_flags", "tile_windows"):
        got = plan.export(name_)
        want = ref[name_]
        assert got.shape == want.shape and np.array_equal(got, want.astype(got.dtype)), name_
    st = plan.stats()
    assert st["tiles"] == ref["win_tile_ptr"][-1]
    assert st["dup_windows"] == int(ref["win_dup"].sum())
    if "bsb_smem_edges" in kw:
        assert st["large_windows"] > 0


def test_bucket_counts_without_lists():
    """Default plans count the rows of each degree bucket (stats and the
    bucket offsets) but build the per-bucket row lists only on request."""
    ensure_built()
    g = graphgen.powerlaw(num_nodes=20000, seed=4)
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 2, 32, "bf16", bucket_bounds=(4, 16, 128))
    ref = ref_planner.degree_buckets(g.row_ptr, (4, 16, 128))
    assert np.array_equal(plan.export("bucket_ptr"), ref["bucket_ptr"])
    assert plan.stats()["bucket_count"] == list(np.diff(ref["bucket_ptr"]))
    with pytest.raises(g3s.G3SError) as ei:
        plan.export("bucket_rows")
    assert ei.value.status == 2
    a = g3s.workspace_size(g.num_nodes, g.num_edges, 2, 32, "bf16")
    b = g3s.workspace_size(g.num_nodes, g.num_edges, 2, 32, "bf16", degree_buckets=1)
    assert b >= a + 5 * g.num_nodes


def test_planner_default_heavy_threshold():
    """Default options: the heavy-row threshold is ten times the mean degree
    in [64, 512], chunks of 512, and the heavy rows and chunks equal the
    reference planner's for that threshold."""
    ensure_built()
    graphs = [graphgen.powerlaw(num_nodes=20_000, seed=41),                      # mean 14: 143
              graphgen.lognormal_local(num_nodes=20_000, radius=512, seed=42),    # mean 50: ~504
              graphgen.tiny_poisson(seed=43),                                     # no heavy row
              graphgen.random_csr(300, 3, seed=44, zero_frac=0.5)]                # mean < 6.4: 64
    for g in graphs:
        rp, ci = upload_graph(g)
        plan = g3s.Plan(rp, ci, g.num_nodes, 1, 64, "f16")
        st = plan.stats()
        t = ref_planner.auto_heavy_threshold(g.num_nodes, g.num_edges)
        assert st["heavy_threshold"] == t and st["chunk_edges"] == 512
        ref = ref_planner.heavy_chunks(g.row_ptr, t, 512)
        for name_ in ("heavy_rows", "heavy_chunk_ptr", "chunks"):
            got = plan.export(name_)
            assert np.array_equal(got, ref[name_].astype(got.dtype)), name_
    assert ref_planner.auto_heavy_threshold(20_000, 285_200) == 143


# ---------------------------------------------------------------------------
# errors
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["col_out_of_range", "negative_col", "row_ptr_decreasing", "row_ptr_end",
                                  "row_ptr_start"])
def test_bad_graph_is_rejected(case):
    ensure_built()
    rp = np.array([0, 2, 4, 5], np.int32)
    col = np.array([1, 2, 0, 2, 1], np.int32)
    if case == "col_out_of_range":
        col[3] = 3
    elif case == "negative_col":
        col[0] = -1
    elif case == "row_ptr_decreasing":
        rp[1], rp[2] = 4, 2
    elif case == "row_ptr_end":
        rp[3] = 4
    elif case == "row_ptr_start":
        rp[0] = 1
    r, c = upload_graph(graphgen.Graph(rp, col))
    with pytest.raises(g3s.G3SError) as ei:
        g3s.Plan(r, c, 3, 1, 16, "f32")
    assert ei.value.status == 3


def test_argument_errors():
    ensure_built()
    g = graphgen.tiny_poisson(num_nodes=64)
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 8, 32, "bf16")
    dev = device()
    buf = torch.zeros(g.num_nodes * 256 + 8, dtype=torch.bfloat16, device=dev)
    good = buf[:g.num_nodes * 256]
    bad = buf[2:2 + g.num_nodes * 256]  # 4-byte offset: not 16-byte aligned
    lib = g3s.load_library()
    s = torch.cuda.current_stream().cuda_stream
    h = plan.handle
    assert lib.g3s_forward(h, bad.data_ptr(), good.data_ptr(), good.data_ptr(), None, good.data_ptr(), None, s) == 1
    assert lib.g3s_forward(h, good.data_ptr(), good.data_ptr(), good.data_ptr(), good.data_ptr(), good.data_ptr(),
                           None, s) == 1  # Eproj on a standard plan
    assert lib.g3s_forward(h, None, good.data_ptr(), good.data_ptr(), None, good.data_ptr(), None, s) == 1
    with pytest.raises(TypeError):
        plan.forward(good.float(), good.float(), good.float())
    # too small a workspace
    o = g3s.default_options()
    out = ctypes.c_void_p()
    ws = torch.empty(1024, dtype=torch.uint8, device=dev)
    assert lib.g3s_plan_create(rp.data_ptr(), ci.data_ptr(), g.num_nodes, g.num_edges, 8, 32, 2, 0, ctypes.byref(o),
                               ws.data_ptr(), 1024, s, ctypes.byref(out)) == 4


def test_repeated_persistent_launches():
    """Forwards and aggregations on one plan, back to back in the persistent
    launch form (the work queue reused): every repeat gives the first one's
    bits."""
    ensure_built()
    g = graphgen.lognormal_local(num_nodes=120_000, radius=1024, seed=61)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 4, 32, False, seed=62)
    t = {k: v.to(device()) for k, v in cast_values(vals, "bf16").items()}
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 4, 32, "bf16")
    W = torch.ones(g.num_edges, 4, dtype=torch.bfloat16, device=device())
    first = plan.forward(t["Q"], t["K"], t["V"]).clone()
    agg0 = plan.aggregate(W, t["V"], normalize=True).clone()
    for _ in range(3):
        assert torch.equal(plan.forward(t["Q"], t["K"], t["V"]), first)
        assert torch.equal(plan.aggregate(W, t["V"], normalize=True), agg0)
    plan.check()
    rows = np.random.default_rng(63).choice(g.num_nodes, 2000, replace=False)
    want = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, 4, 32, "bf16", "standard",
                          *(cast_values(vals, "bf16")[k] for k in "QKV"), rows=rows)
    assert_close(first[torch.from_numpy(rows).to(device())], want, "bf16", "O")
