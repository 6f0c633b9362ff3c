"""g3s_forward_noalloc: the fused forward for callers that cannot allocate
device memory (engines that hand out memory only at build time, processes
whose GPU memory is held by another allocator, fixed memory budgets).

It must give the same answer as the usual plan + forward path and as the
fp64 oracle, within the tolerances of the other GPU tests, on two calls in a
row (the second call reuses the static scratch the first one left behind),
and across calls on different graphs and shapes (each call carves the shared
scratch afresh, so partial results and chunk lists move between calls).
Kept in a file of its own that pytest collects last.
"""
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, cast_values, device, ensure_built, upload_graph

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, rp, ci, g, w, t, O, Eout):
    Q, K, V = (t[k] for k in "QKV")
    E = t.get("E")
    return lib.g3s_forward_noalloc(rp.data_ptr(), ci.data_ptr(), g.num_nodes, g.num_edges, w["H"], w["d"],
                                   g3s.DTYPES[w["dtype"]], g3s.VARIANTS[w["variant"]], Q.data_ptr(), K.data_ptr(),
                                   V.data_ptr(), E.data_ptr() if E is not None else None, O.data_ptr(),
                                   Eout.data_ptr() if Eout is not None else None,
                                   torch.cuda.current_stream().cuda_stream)


CASES = {
    # every case has heavy rows, so partial results go through the static scratch
    "powerlaw_f16": (lambda: graphgen.powerlaw(num_nodes=6000, max_degree=3000, seed=41),
                     dict(H=1, d=64, dtype="f16", variant="standard")),
    "lognormal_bf16": (lambda: graphgen.lognormal_local(num_nodes=20000, radius=1024, seed=42),
                       dict(H=4, d=32, dtype="bf16", variant="standard")),
    # the RTMScore form over a graph with heavy rows: plain-sum partials and Eout
    "rtmscore_powerlaw_f32": (lambda: graphgen.powerlaw(num_nodes=4000, max_degree=2500, seed=43),
                              dict(H=8, d=16, dtype="f32", variant="rtmscore")),
    # the RTMScore workload's shape (16 in-edges per node, no heavy row)
    "rtmscore_batch_f32": (lambda: graphgen.rtmscore_batch(num_graphs=3, min_nodes=40, max_nodes=90, seed=44),
                           dict(H=8, d=16, dtype="f32", variant="rtmscore")),
}


class _Case:
    """A graph and its inputs on the device, the oracle's answer, and the usual path's."""

    def __init__(self, name):
        make_graph, w = CASES[name]
        self.name, self.w = name, w
        g = self.g = make_graph()
        rtm = self.rtm = w["variant"] == "rtmscore"
        vals = graphgen.make_values(g.num_nodes, g.num_edges, w["H"], w["d"], rtm, seed=45)
        host = cast_values(vals, w["dtype"])
        dev = device()
        self.rp, self.ci = upload_graph(g)
        self.t = {k: v.to(dev) for k, v in host.items()}
        res = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, w["H"], w["d"], w["dtype"], w["variant"],
                             host["Q"], host["K"], host["V"], host.get("E"), want_eout=rtm)
        self.O_star, self.E_star = res if rtm else (res, None)
        plan = g3s.Plan(self.rp, self.ci, g.num_nodes, w["H"], w["d"], w["dtype"], w["variant"])
        if rtm:
            O_ref, E_ref = plan.forward(self.t["Q"], self.t["K"], self.t["V"], self.t["E"], want_eout=True)
        else:
            O_ref, E_ref = plan.forward(self.t["Q"], self.t["K"], self.t["V"]), None
        torch.cuda.synchronize()
        self.chunks = plan.stats()["chunks"]
        self.O_ref = O_ref.double().cpu().numpy()
        self.E_ref = E_ref.double().cpu().numpy() if rtm else None

    def call_and_check(self, lib, label):
        g, w, dev = self.g, self.w, device()
        O = torch.full((g.num_nodes, w["H"], w["d"]), float("nan"), dtype=torch.float32, device=dev)
        Eout = torch.full((g.num_edges, w["H"], w["d"]), float("nan"), dtype=torch.float32, device=dev) \
            if self.rtm else None
        st = _noalloc_call(lib, self.rp, self.ci, g, w, self.t, O, Eout)
        assert st == 0, lib.g3s_last_error().decode()
        torch.cuda.synchronize()
        assert_close(O, self.O_star, w["dtype"], "O vs oracle (%s, %s)" % (self.name, label))
        assert_close(O, self.O_ref, w["dtype"], "O vs g3s_forward (%s, %s)" % (self.name, label))
        if self.rtm:
            assert_close(Eout, self.E_star, w["dtype"], "Eout vs oracle (%s, %s)" % (self.name, label))
            assert_close(Eout, self.E_ref, w["dtype"], "Eout vs g3s_forward (%s, %s)" % (self.name, label))


def _require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle_and_plan_forward_twice(name):
    _require_gpu()
    case = _Case(name)
    if name != "rtmscore_batch_f32":
        assert case.chunks > 0, "case must exercise the heavy-row scratch"
    lib = g3s.load_library()
    for call in range(2):
        case.call_and_check(lib, "call %d" % call)


def test_noalloc_alternating_graphs():
    """Calls on different graphs, shapes and forms in turn: the scratch's
    carve layout, chunk lists and partials move between calls, and each
    result still matches the oracle and the usual path."""
    _require_gpu()
    cases = {n: _Case(n) for n in ("powerlaw_f16", "rtmscore_powerlaw_f32", "lognormal_bf16",
                                   "rtmscore_batch_f32")}
    lib = g3s.load_library()
    order = ["powerlaw_f16", "rtmscore_powerlaw_f32", "powerlaw_f16", "lognormal_bf16", "rtmscore_batch_f32",
             "rtmscore_powerlaw_f32", "lognormal_bf16", "powerlaw_f16"]
    for i, n in enumerate(order):
        cases[n].call_and_check(lib, "step %d" % i)


def test_noalloc_rejects_graph_beyond_scratch():
    """A plan larger than the static scratch is refused before any device work."""
    _require_gpu()
    lib = g3s.load_library()
    n, e = 4_000_000, 200_000_000  # ~9 B per node alone exceeds the scratch
    st = lib.g3s_forward_noalloc(None, None, n, e, 4, 32, g3s.DTYPES["bf16"], 0, None, None, None, None, None,
                                 None, torch.cuda.current_stream().cuda_stream)
    assert st == 4 and b"static scratch" in lib.g3s_last_error()
