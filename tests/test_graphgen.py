"""Structure of the synthetic workloads (CPU)."""
import numpy as np
import pytest

import graphgen


def _check_csr(g, self_loops_allowed=False):
    rp = g.row_ptr.astype(np.int64)
    assert rp[0] == 0 and np.all(np.diff(rp) >= 0) and rp[-1] == g.num_edges
    c = g.col_idx.astype(np.int64)
    assert c.min(initial=0) >= 0 and c.max(initial=0) < g.num_nodes
    rows = np.repeat(np.arange(g.num_nodes), np.diff(rp))
    key = rows * g.num_nodes + c
    assert np.all(np.diff(key) > 0), "sources must be distinct and ascending per row"
    if not self_loops_allowed:
        assert not np.any(rows == c)
    return rows, c


@pytest.mark.parametrize("name", list(graphgen.WORKLOADS))
def test_small_workloads_are_valid_and_seeded(name):
    g1, v1, w = graphgen.make_workload(name, "small")
    g2, v2, _ = graphgen.make_workload(name, "small")
    assert np.array_equal(g1.row_ptr, g2.row_ptr) and np.array_equal(g1.col_idx, g2.col_idx)
    assert all(np.array_equal(v1[k], v2[k]) for k in v1)
    _check_csr(g1, self_loops_allowed=name in ("batched_dense", "batched_complete", "clustered_heavy"))
    assert v1["Q"].shape == (g1.num_nodes, w.heads, w.head_dim)
    if w.variant == "rtmscore":
        assert v1["E"].shape == (g1.num_edges, w.heads, w.head_dim)


def test_tiny_full():
    g = graphgen.tiny_poisson()
    _check_csr(g)
    assert g.num_nodes == 320 and 12 < g.degrees().mean() < 16


def test_rtmscore_full():
    g = graphgen.rtmscore_batch()
    rows, c = _check_csr(g)
    assert np.all(g.degrees() == 16) and 64 * 200 <= g.num_nodes <= 64 * 600


def test_batched_dense_full():
    g = graphgen.batched_dense()
    rows, c = _check_csr(g, self_loops_allowed=True)
    assert np.sum(rows == c) == g.num_nodes  # one self loop per node
    # off-diagonal density close to 0.3 within graphs of U[20,60] nodes
    assert 12 < g.degrees().mean() < 16


def test_batched_complete_is_complete():
    """Every graph of the batch is complete with self loops: each row lists all
    nodes of its own graph."""
    g = graphgen.make_workload("batched_complete", "small")[0]
    rows, c = _check_csr(g, self_loops_allowed=True)
    deg = g.degrees()
    start = 0
    while start < g.num_nodes:  # a graph is a run of rows with the same degree = its size
        n = int(deg[start])
        assert np.all(deg[start:start + n] == n)
        for r in range(start, start + n):
            assert np.array_equal(c[g.row_ptr[r]:g.row_ptr[r + 1]], np.arange(start, start + n))
        start += n


def test_lognormal_local_small_structure():
    g = graphgen.lognormal_local(num_nodes=50_000, seed=77)
    rows, c = _check_csr(g)
    off = np.abs(c - rows)
    local = np.mean(off <= 4096)
    expect = 0.6 + 0.4 * 8192 / g.num_nodes  # local draws plus uniform draws that land near
    assert abs(local - expect) < 0.01
    assert 45 < g.degrees().mean() < 56


def test_powerlaw_small_structure():
    g = graphgen.powerlaw(num_nodes=20_000, seed=78)
    _check_csr(g)
    d = g.degrees()
    assert 13 < d.mean() < 15.5 and d.max() > 500


def test_clustered_heavy_full():
    """Heavy rows take 1024 distinct sources from their window's pool of 2048,
    light rows 8 uniform ones, about 3 : 1."""
    g = graphgen.clustered_heavy()
    _check_csr(g, self_loops_allowed=True)
    deg = g.degrees()
    assert g.num_nodes == 16384 and set(np.unique(deg)) == {8, 1024}
    assert 0.7 < np.mean(deg == 1024) < 0.8
    w = 37
    heavy_rows = [r for r in range(16 * w, 16 * w + 16) if deg[r] == 1024]
    pool = np.unique(np.concatenate([g.col_idx[g.row_ptr[r]:g.row_ptr[r + 1]] for r in heavy_rows]))
    assert pool.size <= 2048
