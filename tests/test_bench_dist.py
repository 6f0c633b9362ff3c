"""bench.py's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, and the whole-job rate counts every replica."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        with open(os.path.join(out_dir, "rank%d" % rank), "w") as f:
            f.write(repr(t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [float(open(tmp_path / ("rank%d" % r)).read()) for r in range(2)]
    assert got == [15.0, 15.0]


def test_single_process_paths():
    assert bench.max_over_ranks(3.5) == 3.5
    # 100 edges x 10 steps x 4 replicas in 2 ms
    assert bench.whole_job_rate(100, 10, 4, 2.0) == pytest.approx(2.0e6)


def test_byte_model():
    import graphgen

    g = graphgen.tiny_poisson()
    w = graphgen.WORKLOADS["tiny_poisson"]
    gathered, compulsory = bench.byte_counts(g, w, "f32")
    hd = w.heads * w.head_dim
    assert gathered == 4 * (g.num_nodes + 1) + 4 * g.num_edges + 2 * g.num_nodes * hd * 4 + 2 * g.num_edges * hd * 4
    assert compulsory == 4 * (g.num_nodes + 1) + 4 * g.num_edges + 4 * g.num_nodes * hd * 4


def test_aggregate_byte_model():
    import graphgen

    g = graphgen.tiny_poisson()
    w = graphgen.WORKLOADS["tiny_poisson"]
    gathered, compulsory = bench.aggregate_bytes(g, w, "f32")
    n, e, h, hd = g.num_nodes, g.num_edges, w.heads, w.heads * w.head_dim
    csr = 4 * (n + 1) + 4 * e
    # per edge: its H weights and its source's H*d features; O once
    assert gathered == csr + e * h * 4 + e * hd * 4 + n * hd * 4
    assert compulsory == csr + e * h * 4 + n * hd * 4 + n * hd * 4


def test_kernel_hash_ignores_comments(tmp_path, monkeypatch):
    """The DRAM-traffic record stays valid across comment edits of the CUDA
    sources and is voided by any code edit."""
    csrc = tmp_path / "sparse_graph_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    f.write_text('__global__ void k(int* p) { p[0] = 1; }  // one\n/* block */\nconst char* s = "a//b";\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_sources_hash()
    f.write_text('// header\n__global__ void k(int* p) { p[0] = 1; }  // two\n\nconst char* s = "a//b";\n')
    assert bench.kernel_sources_hash() == h0
    f.write_text('__global__ void k(int* p) { p[0] = 2; }\nconst char* s = "a//b";\n')
    assert bench.kernel_sources_hash() != h0
    f.write_text('__global__ void k(int* p) { p[0] = 1; }\nconst char* s = "a//c";\n')
    assert bench.kernel_sources_hash() != h0


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the reference arm (the oracle on the host cores) runs
    and prints on rank 0 alone; another rank exits 0 without output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_poisson", "--size", "small",
           "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == "", r.stderr
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny_poisson"


def test_tile_item_flop_count():
    """Issued tensor FLOPs of tile items, counted by hand: a pair of windows of
    5 and 3 tiles (units 3 and 2) is S^T = 128 x 32 x d and O^T = 128 x 16 x 16
    per unit of each window; a single window of 16 tiles (8 units) is
    128 x 16 x d and 8 units; a split-window slice (flag bit 16 or 17) counts
    as a single window of its tiles."""
    d, H = 64, 8
    pair = [10, 0, 5, 2 | (3 << 8), 11, 5, 3, 0]
    single = [12, 8, 16, 1 | (8 << 8), 0, 0, 0, 0]
    slice_ = [13, 24, 7, 1 | (4 << 8) | (1 << 17), 0, 3, 0, 0]
    want_pair = 2 * 128 * 32 * d + 2 * 128 * 16 * 16 * (3 + 2)
    want_single = 2 * 128 * 16 * d + 2 * 128 * 16 * 16 * 8
    want_slice = 2 * 128 * 16 * d + 2 * 128 * 16 * 16 * 4
    assert bench.items_mma_flops([pair], H, d) == H * want_pair
    assert bench.items_mma_flops([pair, single, slice_], H, d) == H * (want_pair + want_single + want_slice)
    assert bench.items_mma_flops([], H, d) == 0
