"""g3s_gather_probe reads exactly the rows it reports: the XOR of every word
it read (combined over the warps' sink words) equals the XOR of the words of
the rows of the documented hashed sequence, j < rows read, computed on the
host."""
import numpy as np
import pytest
import torch

import sparse_graph_attention_gb300 as g3s

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("plain", [False, True])
@pytest.mark.parametrize("row_bytes", [16, 128, 512, 1024, 4096])
def test_gather_probe_reads_the_listed_rows(row_bytes, plain):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()
    rng = np.random.default_rng(row_bytes)
    rows = 256
    words = row_bytes // 4
    src_h = rng.integers(0, 2 ** 31, size=rows * words, dtype=np.int64).astype(np.int32)
    src = torch.from_numpy(src_h).cuda()
    ctas = 3
    sink = torch.zeros(ctas * 8, dtype=torch.int32, device="cuda")
    n = g3s.gather_probe(src, row_bytes, 5000, ctas, sink, plain)
    torch.cuda.synchronize()
    assert n >= 5000
    j = np.arange(n, dtype=np.uint64) + np.uint64(1)
    with np.errstate(over="ignore"):
        r = (j * np.uint64(0x9E3779B97F4A7C15)) >> np.uint64(64 - 8)
    row_xor = np.bitwise_xor.reduce(src_h.reshape(rows, words).view(np.uint32), axis=1)
    want = np.bitwise_xor.reduce(row_xor[r.astype(np.int64)])
    got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
    assert got == want
