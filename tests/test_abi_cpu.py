"""libg3s loads, exports every symbol include/g3s.h declares, and its host-side
argument checks answer without touching a GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_graph_attention_gb300 as g3s
from sparse_graph_attention_gb300 import build as g3s_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "g3s.h")


@pytest.fixture(scope="module")
def lib():
    g3s_build.build()
    return g3s.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(g3s_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", g3s.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (g3s_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(lib, n)  # resolvable through ctypes
    assert sorted(g3s.EXPORTED) == names


def test_struct_layout_matches_c(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "g3s.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(g3s_plan_options), offsetof(g3s_plan_options, rtm_epsilon),
         sizeof(g3s_plan_stats), offsetof(g3s_plan_stats, workspace_used));
  return 0;
}''')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.dirname(HEADER), str(prog), "-o", str(exe)])
    c = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    py = [ctypes.sizeof(g3s.PlanOptions), g3s.PlanOptions.rtm_epsilon.offset,
          ctypes.sizeof(g3s.PlanStats), g3s.PlanStats.workspace_used.offset]
    assert c == py


def test_version_and_status_strings(lib):
    assert g3s.version().startswith("g3s")
    assert lib.g3s_status_string(0) == b"G3S_OK"
    assert lib.g3s_status_string(3) == b"G3S_ERR_BAD_GRAPH"
    assert lib.g3s_status_string(99) == b"G3S_ERR_UNKNOWN"


def test_default_options(lib):
    o = g3s.default_options()
    assert list(o.bucket_bounds) == [32, 256, 2048]
    assert o.heavy_threshold == 0 and o.chunk_edges == 0 and o.validate_graph == 1
    assert o.tile_density_milli == 100 and o.tile_pool_density_milli == 180 and o.tile_max_tiles == 16 \
        and o.out_dtype == 0
    assert abs(o.rtm_epsilon - 1e-6) < 1e-12 and o.rtm_elementwise_clamp == 1
    assert o.pack_rows == -1 and o.degree_buckets == 0 and o.small_graph_rows == 1024
    assert o.tile_split_density_milli == 150 and o.tile_split_parallel == 0


@pytest.mark.parametrize("args,status", [
    ((100, 1000, 4, 32, "bf16"), 0),
    ((100, 1000, 4, 48, "bf16"), 2),     # head_dim not supported
    ((100, 1000, 3, 32, "bf16"), 2),     # H*d*2 = 192 B not a power of two
    ((-1, 1000, 4, 32, "bf16"), 1),      # negative N
    ((100, 2**31, 4, 32, "bf16"), 1),    # E overflows int32
    ((100, 1000, 0, 32, "f32"), 1),      # no heads
])
def test_workspace_size_checks(lib, args, status):
    if status == 0:
        assert g3s.workspace_size(*args) > 0
    else:
        with pytest.raises(g3s.G3SError) as ei:
            g3s.workspace_size(*args)
        assert ei.value.status == status


def test_workspace_grows_with_bsb(lib):
    a = g3s.workspace_size(10_000, 500_000, 4, 32, "bf16", bsb=0)
    b = g3s.workspace_size(10_000, 500_000, 4, 32, "bf16", bsb=1)
    assert b > a


def test_bad_options_rejected(lib):
    for kw in (dict(bucket_bounds=[10, 5, 20]), dict(heavy_threshold=-1), dict(chunk_edges=-1),
               dict(bsb_smem_edges=100000), dict(tile_path=2), dict(pack_rows=2), dict(tile_pool_density_milli=-1),
               dict(degree_buckets=2), dict(small_graph_rows=-1), dict(tile_split_density_milli=-1),
               dict(tile_split_density_milli=99), dict(tile_split_density_milli=1001),
               dict(tile_split_parallel=2), dict(tile_split_parallel=-1)):
        with pytest.raises(g3s.G3SError) as ei:
            g3s.workspace_size(100, 1000, 4, 32, "bf16", **kw)
        assert ei.value.status == 1


def test_workspace_of_split_windows(lib):
    """The partial states of edge-parallel split windows are workspace only
    where the tile path can run (fp16/bf16, d = 64, standard form), bounded by
    the split density: 2000 E / (128 split_milli) partial rows of 4 H (d + 2)
    bytes; node-parallel chains need none."""
    args = (10_000, 500_000, 8, 64, "bf16")
    off = g3s.workspace_size(*args, tile_split_density_milli=0)
    edge = g3s.workspace_size(*args, tile_split_parallel=1)
    dense = g3s.workspace_size(*args, tile_split_parallel=1, tile_split_density_milli=1000)
    node = g3s.workspace_size(*args)
    rows = 2000 * 500_000 // (128 * 150) + 16
    assert edge - off >= rows * 4 * 8 * 66 and edge > dense > off
    assert off < node < off + rows * 4 * 8 * 66 // 10
    assert g3s.workspace_size(10_000, 500_000, 4, 32, "bf16") == \
        g3s.workspace_size(10_000, 500_000, 4, 32, "bf16", tile_split_density_milli=0)


def test_calls_without_plan_fail_cleanly(lib):
    P = ctypes.c_void_p
    assert lib.g3s_forward(None, None, None, None, None, None, None, None) == 1
    assert b"NULL plan" in lib.g3s_last_error()
    st = g3s.PlanStats()
    assert lib.g3s_plan_get_stats(None, ctypes.byref(st)) == 1
    assert lib.g3s_plan_export(None, 0, None, 0, None) == 1
    lib.g3s_plan_destroy(None)
    out = P()
    o = g3s.default_options()
    # NULL workspace and misaligned workspace are rejected before any CUDA call
    assert lib.g3s_plan_create(P(16), P(16), 10, 20, 1, 16, 0, 0, ctypes.byref(o), None, 0, None,
                               ctypes.byref(out)) == 4
    assert lib.g3s_plan_create(P(16), P(16), 10, 20, 1, 16, 0, 0, ctypes.byref(o), P(4096 + 8), 1 << 30, None,
                               ctypes.byref(out)) == 4
    assert lib.g3s_plan_create(None, P(16), 10, 20, 1, 16, 0, 0, ctypes.byref(o), P(4096), 1 << 30, None,
                               ctypes.byref(out)) == 1


def test_noalloc_rejects_graphs_beyond_its_scratch(lib):
    """The static-scratch entry point refuses, before touching the GPU, a graph
    whose plan would not fit in its built-in scratch."""
    P = ctypes.c_void_p
    n, e = 2_000_000, 100_000_000
    assert g3s.workspace_size(n, e, 4, 32, "bf16", bsb=0) > g3s.NOALLOC_SCRATCH_BYTES
    st = lib.g3s_forward_noalloc(P(256), P(256), n, e, 4, 32, 2, 0, P(256), P(256), P(256), None, P(256), None,
                                 None)
    assert st == 4
    assert b"static scratch" in lib.g3s_last_error()
    assert g3s.workspace_size(200_000, 2_850_000, 1, 64, "f16", bsb=0) <= g3s.NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("n,e", [(320, 4480), (200_000, 2_851_788), (2_000_000, 100_717_572), (1000, 10),
                                 (10, 100_000), (0, 0)])
def test_automatic_heavy_threshold_sizes_like_its_value(lib, n, e):
    """heavy_threshold = 0 resolves to ten times the mean degree in [64, 512]
    (512 for an empty graph): the workspace bound equals the one for that
    value given explicitly."""
    from oracle import planner

    t = planner.auto_heavy_threshold(n, e)
    assert 64 <= t <= 512
    assert g3s.workspace_size(n, e, 4, 32, "bf16") == g3s.workspace_size(n, e, 4, 32, "bf16", heavy_threshold=t)
    if 0 < n and 64 < 10 * e / n < 512:
        assert g3s.workspace_size(n, e, 4, 32, "bf16") != g3s.workspace_size(n, e, 4, 32, "bf16", heavy_threshold=t + 7)
