"""Physical edge numbering (g3s_plan_set_edge_ids): edge features and weights
stored in their own order, reached through a CSR-position -> slot vector."""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, device, ensure_built, upload_graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


def _slots(E, extra, seed):
    rng = np.random.default_rng(seed)
    return rng.permutation(E + extra)[:E].astype(np.int32), E + extra


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rtmscore_reads_and_writes_physical_slots(dtype):
    g = graphgen.rtmscore_batch(num_graphs=4, min_nodes=30, max_nodes=70, seed=31)
    H, d = 8, 16
    ids, slots = _slots(g.num_edges, 53, 32)
    rng = np.random.default_rng(33)
    q, k, v = (rng.standard_normal((g.num_nodes, H, d)).astype(np.float32) for _ in range(3))
    e_phys = rng.standard_normal((slots, H, d)).astype(np.float32)
    t = {n: graphgen.to_dtype(a, dtype) for n, a in (("Q", q), ("K", k), ("V", v), ("E", e_phys))}
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, "rtmscore", heavy_threshold=8, chunk_edges=5,
                    small_graph_rows=0)
    plan.set_edge_ids(torch.from_numpy(ids).to(dev), slots)
    Eout = torch.full((slots, H, d), 7.0, dtype=torch.float32, device=dev)
    O, Eout = plan.forward(t["Q"].to(dev), t["K"].to(dev), t["V"].to(dev), t["E"].to(dev), Eout=Eout,
                           want_eout=True)
    torch.cuda.synchronize()
    e_csr = t["E"][torch.from_numpy(ids.astype(np.int64))]
    want_O, want_E = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, H, d, dtype, "rtmscore", t["Q"], t["K"],
                                    t["V"], e_csr, want_eout=True)
    assert_close(O, want_O, dtype, "O")
    assert_close(Eout[torch.from_numpy(ids.astype(np.int64)).to(dev)], want_E, dtype, "Eout")
    untouched = np.setdiff1d(np.arange(slots), ids)
    assert torch.all(Eout[torch.from_numpy(untouched).to(dev)] == 7.0)


def test_aggregate_reads_physical_weights():
    g = graphgen.powerlaw(num_nodes=3000, max_degree=2000, seed=34)
    H, d = 2, 32
    ids, slots = _slots(g.num_edges, 101, 35)
    rng = np.random.default_rng(36)
    x = rng.standard_normal((g.num_nodes, H, d)).astype(np.float32)
    w_phys = (np.abs(rng.standard_normal((slots, H))) + 0.1).astype(np.float32)
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, "f32", heavy_threshold=50, chunk_edges=17,
                    small_graph_rows=0)
    plan.set_edge_ids(torch.from_numpy(ids).to(dev), slots)
    O = plan.aggregate(torch.from_numpy(w_phys).to(dev), torch.from_numpy(x).to(dev), normalize=True)
    torch.cuda.synchronize()
    want = oracle.aggregate(g.row_ptr, g.col_idx, g.num_nodes, H, d, "f32", w_phys[ids], x, normalize=True)
    assert_close(O, want, "f32", "O")
    plan.set_edge_ids(None, 0)  # back to CSR positions
    O2 = plan.aggregate(torch.from_numpy(w_phys[ids]).to(dev), torch.from_numpy(x).to(dev), normalize=True)
    assert_close(O2, want, "f32", "O (CSR order)")


def test_host_path_with_edge_ids():
    g = graphgen.rtmscore_batch(num_graphs=2, min_nodes=30, max_nodes=50, seed=37)
    H, d = 8, 16
    ids, slots = _slots(g.num_edges, 9, 38)
    rng = np.random.default_rng(39)
    t = {n: torch.from_numpy(rng.standard_normal(s).astype(np.float32))
         for n, s in (("Q", (g.num_nodes, H, d)), ("K", (g.num_nodes, H, d)), ("V", (g.num_nodes, H, d)),
                      ("E", (slots, H, d)))}
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, "f32", "rtmscore")
    plan.set_edge_ids(torch.from_numpy(ids).to(dev), slots)
    O, Eout = plan.forward(*(t[n].to(dev) for n in "QKV"), t["E"].to(dev), want_eout=True)
    pin = {n: v.pin_memory() for n, v in t.items()}
    Oh = torch.empty_like(pin["Q"]).pin_memory()
    Eoh = torch.zeros_like(pin["E"]).pin_memory()
    plan.forward_host(pin["Q"], pin["K"], pin["V"], Oh, pin["E"], Eoh)
    torch.cuda.synchronize()
    sel = torch.from_numpy(ids.astype(np.int64))
    assert torch.equal(Oh, O.cpu()) and torch.equal(Eoh[sel], Eout.cpu()[sel])


def test_out_of_range_edge_id_rejected():
    g = graphgen.tiny_poisson(num_nodes=50)
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, 1, 16, "f32", "rtmscore")
    ids = np.arange(g.num_edges, dtype=np.int32)
    ids[7] = g.num_edges  # one past the slots
    with pytest.raises(g3s.G3SError) as ei:
        plan.set_edge_ids(torch.from_numpy(ids).to(dev), g.num_edges)
    assert ei.value.status == 3
    ids[7] = -1
    with pytest.raises(g3s.G3SError):
        plan.set_edge_ids(torch.from_numpy(ids).to(dev), g.num_edges)
