"""GPU parity of g3s_aggregate (weighted, optionally normalised aggregation)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, cast_values, device, ensure_built, upload_graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


def _case(g, H, d, dtype, normalize, positive, seed, plan_kw=None, eps=1e-6):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((g.num_nodes, H, d)).astype(np.float32)
    w = rng.standard_normal((g.num_edges, H)).astype(np.float32)
    if positive:
        w = np.abs(w) + 0.05
    xt, wt = graphgen.to_dtype(x, dtype), graphgen.to_dtype(w, dtype)
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, **(plan_kw or {}))
    O = plan.aggregate(wt.to(device()), xt.to(device()), normalize=normalize, eps=eps)
    torch.cuda.synchronize()
    want = oracle.aggregate(g.row_ptr, g.col_idx, g.num_nodes, H, d, dtype, wt, xt, normalize=normalize, eps=eps)
    assert_close(O, want, dtype, "O (aggregate)")
    return plan


@pytest.mark.parametrize("name", list(graphgen.WORKLOADS))
@pytest.mark.parametrize("normalize", [False, True])
def test_aggregate_small_workloads(name, normalize):
    g, _, w = graphgen.make_workload(name, "small")
    _case(g, w.heads, w.head_dim, w.dtype, normalize, positive=normalize, seed=w.number)


def test_aggregate_popcornbench_shape():
    """The CSR aggregation task's sizes: N = 320, 8 heads x 32, fp32, unnormalised."""
    g = graphgen.tiny_poisson()
    _case(g, 8, 32, "f32", False, positive=False, seed=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_aggregate_heavy_rows(dtype):
    g = graphgen.powerlaw(num_nodes=5000, max_degree=4000, seed=8)
    plan = _case(g, 2, 32, dtype, True, positive=True, seed=9, plan_kw=dict(heavy_threshold=40, chunk_edges=13, small_graph_rows=0))
    assert plan.stats()["chunks"] > 0
    _case(g, 2, 32, dtype, False, positive=False, seed=10, plan_kw=dict(heavy_threshold=40, chunk_edges=13, small_graph_rows=0))


def test_aggregate_full_powerlaw():
    g, _, w = graphgen.make_workload("powerlaw", "full")
    _case(g, w.heads, w.head_dim, w.dtype, True, positive=True, seed=11)


def test_aggregate_on_tile_plan_covers_tile_windows():
    """Rows in tile-path windows are aggregated too (the tile kernel is attention-only)."""
    g = graphgen.batched_dense(num_graphs=20, seed=12)
    plan = _case(g, 2, 64, "bf16", True, positive=True, seed=13, plan_kw=dict(tile_path=1, tile_density_milli=0, tile_pool_density_milli=0))
    assert plan.stats()["tile_windows"] > 0


def test_aggregate_multigraph_and_empty_rows():
    g = graphgen.random_csr(150, 40, seed=14, zero_frac=0.3, multigraph=True, sorted_rows=False)
    _case(g, 4, 16, "f32", True, positive=True, seed=15, eps=0.25)
    _case(g, 4, 16, "f32", False, positive=False, seed=16)


def test_aggregate_argument_errors():
    g = graphgen.tiny_poisson(num_nodes=40)
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 1, 16, "f32")
    lib = g3s.load_library()
    x = torch.zeros(g.num_nodes * 16 + 4, device=device())
    w = torch.zeros(g.num_edges, device=device())
    s = torch.cuda.current_stream().cuda_stream
    assert lib.g3s_aggregate(plan.handle, None, x.data_ptr(), x.data_ptr(), 0, 1e-6, s) == 1
    assert lib.g3s_aggregate(plan.handle, w.data_ptr(), x[1:].data_ptr(), x.data_ptr(), 0, 1e-6, s) == 1
    assert lib.g3s_aggregate(plan.handle, w.data_ptr(), x.data_ptr(), x.data_ptr(), 1, -1.0, s) == 1


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("pack", [0, 1])
def test_aggregate_32_byte_rows(dtype, pack):
    """Rows of 32 bytes (one head of 16 16-bit values): 16 lane groups of
    eight edges make a step of 128 slots, wider than the 64-entry index
    window, so each slot loads its own index; short rows, long rows, heavy
    rows (chunks) and empty rows, with and without short-row packs."""
    rng = np.random.default_rng(21)
    n = 1500
    deg = rng.integers(0, 6, n)
    deg[rng.random(n) < 0.1] = rng.integers(60, 400, 1)[0]
    deg[::97] = 0
    deg[5] = 1200  # a heavy row
    rows = [np.sort(rng.choice(n, int(k), replace=False)) for k in deg]
    rp = np.zeros(n + 1, np.int64)
    rp[1:] = np.cumsum(deg)
    g = graphgen.Graph(rp.astype(np.int32), np.concatenate(rows).astype(np.int32))
    plan = _case(g, 1, 16, dtype, True, positive=True, seed=22, plan_kw=dict(pack_rows=pack, heavy_threshold=500,
                                                                              chunk_edges=130, small_graph_rows=0))
    st = plan.stats()
    assert st["chunks"] > 0 and st["pack_rows"] == pack
    _case(g, 1, 16, dtype, False, positive=False, seed=23, plan_kw=dict(pack_rows=pack))
