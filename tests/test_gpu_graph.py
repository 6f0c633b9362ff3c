"""g3s_forward inside a CUDA graph: the forward only enqueues work on the
caller's stream (a memset of the work counter and kernel launches, no
synchronisation, no allocation), so it can be captured once and replayed.
Replays over new input values (copied into the captured buffers) must match
the oracle, as the eager call does."""
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


@pytest.mark.parametrize("name,kw", [("tiny_poisson", {}), ("rtmscore_batch64", {}),
                                     ("batched_dense", {"tile_path": 1, "tile_density_milli": 200, "tile_pool_density_milli": 0}),
                                     ("powerlaw", {"heavy_threshold": 64, "chunk_edges": 40})])
def test_forward_replays_in_a_cuda_graph(name, kw):
    dev = device()
    g, vals, w = graphgen.make_workload(name, "small")
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant, **kw)
    rtm = w.variant == "rtmscore"
    bufs = {k: v.to(dev) for k, v in cast_values(vals, w.dtype).items()}
    O = torch.empty((g.num_nodes, w.heads, w.head_dim), dtype=torch.float32, device=dev)
    Eout = torch.empty((g.num_edges, w.heads, w.head_dim), dtype=torch.float32, device=dev) if rtm else None

    def fwd():
        plan.forward(bufs["Q"], bufs["K"], bufs["V"], bufs.get("E"), O, Eout)

    fwd()  # first call outside the capture (per-device launch set-up)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fwd()
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    for rep in range(3):
        new = graphgen.make_values(g.num_nodes, g.num_edges, w.heads, w.head_dim, rtm, seed=500 + rep)
        t = cast_values(new, w.dtype)
        for k in bufs:
            bufs[k].copy_(t[k].to(dev))
        O.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        res = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant,
                             t["Q"], t["K"], t["V"], t.get("E"), want_eout=rtm)
        if rtm:
            assert_close(O, res[0], w.dtype, "O (replay %d)" % rep)
            assert_close(Eout, res[1], w.dtype, "Eout (replay %d)" % rep)
        else:
            assert_close(O, res, w.dtype, "O (replay %d)" % rep)
