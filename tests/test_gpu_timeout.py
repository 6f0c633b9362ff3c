"""The device-side timeout path: a bounded wait on a barrier that nothing
completes gives up, the host reads G3S_ERR_TIMEOUT, and the context keeps
working (a forward afterwards still matches the oracle)."""
import time

import pytest
import torch

import graphgen
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import ensure_built, run_case

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()
    g, vals, w = graphgen.make_workload("batched_dense", "small")
    plan, _, _ = run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant,
                          plan_kw=dict(tile_path=1, tile_density_milli=150, tile_pool_density_milli=0))
    lib = g3s.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    st = lib.g3s_selftest_wait_timeout(plan.handle, 50_000_000, stream)  # 50 ms
    dt = time.perf_counter() - t0
    assert st == 6, lib.g3s_last_error()  # G3S_ERR_TIMEOUT
    assert 0.04 < dt < 5.0
    plan.check()  # the flag was cleared
    run_case(g, vals, w.heads, w.head_dim, w.dtype, w.variant, plan_kw=dict(tile_path=1, tile_density_milli=150, tile_pool_density_milli=0))
