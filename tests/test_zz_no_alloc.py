"""g3s_forward_noalloc: the fused forward for callers that cannot allocate
device memory (engines that hand out memory only at build time, processes
whose GPU memory is held by another allocator, fixed memory budgets).

It must give the same answer as the usual plan + forward path, within the
tolerances of the other GPU tests, on two calls in a row (the second call
reuses the static scratch the first one left behind).  Kept in a file of its
own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import graphgen
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, cast_values, device, ensure_built, upload_graph

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, rp, ci, g, w, t, dev, O, Eout):
    Q, K, V = (t[k] for k in "QKV")
    E = t.get("E")
    return lib.g3s_forward_noalloc(rp.data_ptr(), ci.data_ptr(), g.num_nodes, g.num_edges, w["H"], w["d"],
                                   g3s.DTYPES[w["dtype"]], g3s.VARIANTS[w["variant"]], Q.data_ptr(), K.data_ptr(),
                                   V.data_ptr(), E.data_ptr() if E is not None else None, O.data_ptr(),
                                   Eout.data_ptr() if Eout is not None else None,
                                   torch.cuda.current_stream().cuda_stream)


CASES = {
    # heavy rows present, so the partial results go through the static scratch
    "powerlaw_f16": (lambda: graphgen.powerlaw(num_nodes=6000, max_degree=3000, seed=41),
                     dict(H=1, d=64, dtype="f16", variant="standard")),
    "lognormal_bf16": (lambda: graphgen.lognormal_local(num_nodes=20000, radius=1024, seed=42),
                       dict(H=4, d=32, dtype="bf16", variant="standard")),
    "rtmscore_f32": (lambda: graphgen.rtmscore_batch(num_graphs=3, min_nodes=40, max_nodes=90, seed=43),
                     dict(H=8, d=16, dtype="f32", variant="rtmscore")),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_plan_forward_twice(name):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()
    make_graph, w = CASES[name]
    g = make_graph()
    vals = graphgen.make_values(g.num_nodes, g.num_edges, w["H"], w["d"], w["variant"] == "rtmscore", seed=44)
    dev = device()
    rp, ci = upload_graph(g)
    t = {k: v.to(dev) for k, v in cast_values(vals, w["dtype"]).items()}
    rtm = w["variant"] == "rtmscore"

    # the usual path: a plan in a caller workspace, then g3s_forward
    plan = g3s.Plan(rp, ci, g.num_nodes, w["H"], w["d"], w["dtype"], w["variant"])
    if rtm:
        O_ref, E_ref = plan.forward(t["Q"], t["K"], t["V"], t["E"], want_eout=True)
    else:
        O_ref, E_ref = plan.forward(t["Q"], t["K"], t["V"]), None
    torch.cuda.synchronize()
    if not rtm:
        assert plan.stats()["chunks"] > 0, "case must exercise the heavy-row scratch"

    lib = g3s.load_library()
    for call in range(2):
        O = torch.full((g.num_nodes, w["H"], w["d"]), float("nan"), dtype=torch.float32, device=dev)
        Eout = torch.full((g.num_edges, w["H"], w["d"]), float("nan"), dtype=torch.float32, device=dev) \
            if rtm else None
        st = _noalloc_call(lib, rp, ci, g, w, t, dev, O, Eout)
        assert st == 0, lib.g3s_last_error().decode()
        torch.cuda.synchronize()
        assert_close(O, O_ref.double().cpu().numpy(), w["dtype"], "O (call %d)" % call)
        if rtm:
            assert_close(Eout, E_ref.double().cpu().numpy(), w["dtype"], "Eout (call %d)" % call)
