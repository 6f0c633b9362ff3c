"""Plans used from several host threads at once (one plan and one stream per
thread): every thread's results match the fp64 oracle.  The C ABI keeps no
shared mutable host state on the forward path (launch caches are per
thread), so concurrent calls on different plans do not interfere."""
import threading

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


CASES = [("tiny_poisson", dict()), ("powerlaw", dict(num_nodes=20_000)), ("batched_dense", dict(num_graphs=64)),
         ("rtmscore_batch64", dict(num_graphs=4))]


def test_forwards_from_four_threads():
    dev = device()
    jobs = []
    for k, (name, kw) in enumerate(CASES):
        w = graphgen.WORKLOADS[name]
        g = w.graph_fn(**kw)
        vals = graphgen.make_values(g.num_nodes, g.num_edges, w.heads, w.head_dim, w.variant == "rtmscore",
                                    seed=50 + k)
        t = cast_values(vals, w.dtype)
        jobs.append((w, g, t))
    results, errors = [None] * len(jobs), []

    def run(i):
        try:
            w, g, t = jobs[i]
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(s):
                rp, ci = upload_graph(g)
                plan = g3s.Plan(rp, ci, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant)
                args = [t[k].to(dev) for k in ("Q", "K", "V")]
                E = t["E"].to(dev) if w.variant == "rtmscore" else None
                for _ in range(20):
                    out = plan.forward(*args, E) if E is not None else plan.forward(*args)
                s.synchronize()
                plan.check()
                results[i] = out[0] if isinstance(out, tuple) else out
        except Exception as e:  # reported on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (w, g, t), O in zip(jobs, results):
        want = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, w.heads, w.head_dim, w.dtype, w.variant,
                              t["Q"], t["K"], t["V"], t.get("E"))
        assert_close(O, want, w.dtype, "O (%s)" % w.name)
