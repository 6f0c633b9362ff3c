"""GPU parity of the TMA-fed form of the fused kernel (plan option tma_gather,
standard form, fp16/bf16 inputs, node rows of 128, 256 or 512 bytes) against
the fp64 oracle, and against the plain-load kernel on the same plan inputs."""
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


def graph_with_degrees(degs, num_nodes, seed):
    """Simple graph whose row i has degs[i] distinct sources (ascending)."""
    rng = np.random.default_rng(seed)
    cols = [np.sort(rng.choice(num_nodes, int(k), replace=False)) for k in degs]
    row_ptr = np.zeros(len(degs) + 1, np.int64)
    row_ptr[1:] = np.cumsum(degs)
    col = np.concatenate(cols) if len(cols) else np.zeros(0, np.int64)
    return graphgen.Graph(row_ptr.astype(np.int32), col.astype(np.int32))


# every degree around the step sizes (4, 8, 16 edges), the 32-edge window
# slide and the heavy-row threshold
EDGE_DEGREES = [0, 1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 23, 24, 31, 32, 33, 40, 47, 48, 63, 64, 65, 66, 95, 96, 97,
                127, 128, 129, 200, 255, 256, 257, 300, 511, 512]

# (dtype, heads, head_dim): node rows of 128, 256 and 512 bytes, every lane-per-head count
SHAPES = [("bf16", 4, 32), ("f16", 1, 64), ("f16", 4, 16), ("f16", 2, 32), ("bf16", 8, 16), ("bf16", 2, 64),
          ("bf16", 1, 128), ("f16", 16, 16), ("bf16", 8, 32), ("f16", 4, 64), ("bf16", 2, 128)]


def _forward(plan, t, dev):
    O = plan.forward(*(t[k].to(dev) for k in ("Q", "K", "V")))
    torch.cuda.synchronize()
    return O


@pytest.mark.parametrize("dtype,H,d", SHAPES, ids=["%s-%dx%d" % s for s in SHAPES])
def test_tma_matches_oracle_and_plain_loads(dtype, H, d):
    n = 700
    degs = np.array((EDGE_DEGREES * (n // len(EDGE_DEGREES) + 1))[:n])
    np.random.default_rng(1).shuffle(degs)
    g = graph_with_degrees(degs, n, seed=2)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, H, d, False, seed=3)
    plan, O, _ = run_case(g, vals, H, d, dtype, "standard",
                          plan_kw=dict(heavy_threshold=300, chunk_edges=37, tma_gather=1))
    st = plan.stats()
    assert st["tma_gather"] == 1 and st["chunks"] > 0
    dev = device()
    rp, ci = upload_graph(g)
    plain = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, "standard", heavy_threshold=300, chunk_edges=37,
                     tma_gather=0)
    assert plain.stats()["tma_gather"] == 0
    O_plain = _forward(plain, cast_values(vals, dtype), dev)
    # same arithmetic in the same order; allow a last-bit difference from
    # instruction selection
    diff = (O - O_plain).abs().max().item()
    assert diff <= 1e-6 * max(O_plain.abs().max().item(), 1e-30), diff


def test_tma_fresh_tensors_each_forward():
    """The tensor maps follow K and V: forwards on new tensors, and two plans of
    different sizes alternating, all match the oracle."""
    dev = device()
    cases = []
    for seed, n in ((11, 900), (12, 1500)):
        g = graphgen.lognormal_local(num_nodes=n, radius=64, seed=seed)
        rp, ci = upload_graph(g)
        plan = g3s.Plan(rp, ci, n, 4, 32, "bf16", "standard", tma_gather=1)
        assert plan.stats()["tma_gather"] == 1
        cases.append((g, plan))
    for rep in range(3):
        for g, plan in cases:
            vals = graphgen.make_values(g.num_nodes, g.num_edges, 4, 32, False, seed=100 + rep)
            t = cast_values(vals, "bf16")
            O = _forward(plan, t, dev)
            want = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, 4, 32, "bf16", "standard", t["Q"], t["K"],
                                  t["V"], None)
            assert_close(O, want, "bf16")


def test_tma_with_tile_windows():
    """Dense windows on the tensor-core tile path, the rest through the TMA-fed
    kernel, in one forward (H=2, d=64: 256-byte rows)."""
    g = graphgen.batched_dense(num_graphs=40, min_nodes=20, max_nodes=60, seed=21)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 2, 64, False, seed=22)
    plan, _, _ = run_case(g, vals, 2, 64, "bf16", "standard",
                          plan_kw=dict(tile_path=1, tile_density_milli=300, tile_pool_density_milli=0, tma_gather=1))
    st = plan.stats()
    assert st["tma_gather"] == 1 and 0 < st["tile_windows"] < st["windows"]


@pytest.mark.parametrize("name", ["powerlaw", "lognormal_local"])
def test_tma_workloads_sixteen_bit_output(name):
    g, vals, w = graphgen.make_workload(name, "small")
    plan, O, _ = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant,
                          plan_kw=dict(out_dtype=w.dtype, tma_gather=1))
    assert plan.stats()["tma_gather"] == 1


def test_tma_not_used_where_unsupported():
    g = graphgen.random_csr(50, 10, seed=5)
    rp, ci = upload_graph(g)
    for dtype, H, d, variant in (("f32", 2, 32, "standard"), ("bf16", 8, 64, "standard"),
                                 ("bf16", 2, 32, "rtmscore"), ("bf16", 1, 16, "standard")):
        plan = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, variant, tma_gather=1)
        assert plan.stats()["tma_gather"] == 0, (dtype, H, d, variant)
    plan = g3s.Plan(rp, ci, g.num_nodes, 4, 32, "bf16", "standard")
    assert plan.stats()["tma_gather"] == 0  # off by default
