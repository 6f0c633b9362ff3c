"""include/g3s.h is a C header: a C99 program built against it alone (gcc
-std=c99 -Wall -Wextra -Werror) links to libg3s.so and gets the same
answers as the Python binding from the entry points that need no GPU (CPU)."""
import ctypes
import os
import shutil
import subprocess

import pytest

import sparse_graph_attention_gb300 as g3s
from sparse_graph_attention_gb300 import build as g3s_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    g3s_build.build()
    exe = str(tmp_path_factory.mktemp("cabi") / "abi_check")
    libdir = os.path.dirname(g3s.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "abi_check.c"), "-L", libdir, "-lg3s", "-Wl,-rpath," + libdir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_matches_binding(program):
    r = subprocess.run([program], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    lib = g3s.load_library()
    assert out["version"] == lib.g3s_version().decode()
    st, n = out["headline"].split()
    assert st == "G3S_OK" and int(n) == g3s.workspace_size(2000000, 100717572, 4, 32, "bf16")
    st, n = out["batched"].split()
    assert st == "G3S_OK" and int(n) == g3s.workspace_size(40851, 560593, 8, 64, "bf16")
    assert out["bad_head_dim"] == "G3S_ERR_UNSUPPORTED"
    assert "head_dim 48" in out["error_detail"]
    so, ss = (int(x) for x in out["struct_sizes"].split())
    assert so == ctypes.sizeof(g3s.PlanOptions) and ss == ctypes.sizeof(g3s.PlanStats)
    o = g3s.default_options()
    assert [int(x) for x in out["defaults"].split()] == [o.tile_density_milli, o.tile_pool_density_milli,
                                                         o.tile_split_density_milli, o.tile_split_parallel,
                                                         o.small_graph_rows]
