"""The small-graph flavour (one CTA per row, its eight warps' partial softmax
states merged in shared memory): parity with the oracle for every form,
input and output type, rows from empty to far past the heavy-row threshold,
and the size limit."""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, cast_values, device, ensure_built, run_case, upload_graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


def _graph(n, seed, degrees=(0, 1, 2, 7, 8, 9, 15, 16, 17, 63, 64, 65, 200, 700)):
    """n rows cycling through the given in-degrees (distinct sources)."""
    rng = np.random.default_rng(seed)
    deg = np.array([degrees[i % len(degrees)] for i in range(n)], np.int64)
    deg = np.minimum(deg, n)
    cols = [np.sort(rng.choice(n, size=d, replace=False)) for d in deg]
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    return graphgen.Graph(rp, np.concatenate(cols).astype(np.int32))


CASES = [("f32", 8, 32, "standard"), ("bf16", 4, 32, "standard"), ("f16", 1, 64, "standard"),
         ("bf16", 8, 64, "standard"), ("f32", 8, 16, "rtmscore"), ("f16", 2, 16, "rtmscore"),
         ("f32", 8, 128, "standard"), ("bf16", 2, 128, "rtmscore")]


@pytest.mark.parametrize("dtype,H,d,variant", CASES, ids=["%s-%dx%d-%s" % c for c in CASES])
def test_small_graph_matches_oracle(dtype, H, d, variant):
    g = _graph(900, seed=H * d)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, d, variant == "rtmscore", seed=d)
    plan, _, _ = run_case(g, vals, H, d, dtype, variant, plan_kw=dict(bsb=0))
    st = plan.stats()
    assert st["small_graph"] == 1 and st["heavy_rows"] > 0  # heavy rows, done without chunks


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_small_graph_sixteen_bit_output(dtype):
    g = _graph(500, seed=3)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 4, 32, False, seed=4)
    plan, O, _ = run_case(g, vals, 4, 32, dtype, "standard", plan_kw=dict(out_dtype=dtype))
    assert plan.stats()["small_graph"] == 1 and O.dtype == g3s.torch_dtype(dtype)


def test_small_graph_limit():
    """1024 rows take the small flavour, 1025 the usual kernel; the option
    moves the limit and 0 turns it off; both give the oracle's result."""
    for n, kw, small in ((1024, {}, 1), (1025, {}, 0), (1025, dict(small_graph_rows=2000), 1),
                         (300, dict(small_graph_rows=0), 0)):
        g = _graph(n, seed=n, degrees=(3, 30, 90))
        vals = graphgen.make_values(n, g.num_edges, 2, 32, False, seed=5)
        plan, _, _ = run_case(g, vals, 2, 32, "bf16", "standard", plan_kw=kw)
        assert plan.stats()["small_graph"] == small, (n, kw)


@pytest.mark.parametrize("normalize", [True, False])
def test_small_graph_aggregate(normalize):
    g = _graph(700, seed=8)
    H, d = 4, 32
    dev = device()
    rp, ci = upload_graph(g)
    rng = np.random.default_rng(9)
    X = graphgen.to_dtype(rng.standard_normal((g.num_nodes, H, d)).astype(np.float32), "f32")
    W = graphgen.to_dtype((rng.random((g.num_edges, H)) + 0.05).astype(np.float32), "f32")
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, "f32")
    assert plan.stats()["small_graph"] == 1
    O = plan.aggregate(W.to(dev), X.to(dev), normalize=normalize)
    want = oracle.aggregate(g.row_ptr, g.col_idx, g.num_nodes, H, d, "f32", W, X, normalize=normalize)
    assert_close(O, want, "f32", "aggregate")


def test_small_graph_deterministic_and_empty():
    g = _graph(257, seed=11)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 8, 32, False, seed=12)
    t = {k: v.to(device()) for k, v in cast_values(vals, "f32").items()}
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 8, 32, "f32")
    a = plan.forward(t["Q"], t["K"], t["V"]).clone()
    b = plan.forward(t["Q"], t["K"], t["V"])
    assert torch.equal(a, b)
    zero_rows = np.flatnonzero(g.degrees() == 0)
    assert zero_rows.size and torch.count_nonzero(a[torch.from_numpy(zero_rows).to(device())]).item() == 0
