"""GPU parity of the tensor-core projection (g3s_linear) and of the layer
entry point (projection + fused forward, g3s_layer_forward) against the fp64
oracle.

Tolerance of the projection, from its arithmetic: the products of 16-bit
values are exact in fp32, the K-term sums are accumulated in fp32, so
|y - y*| <= gamma_K * sum_k |x_k w_k| with gamma_K = K u / (1 - K u),
u = 2^-24; the test allows twice that (an accumulator that truncates instead
of rounding doubles u).  A 16-bit output adds its own rounding, at most
u16 |y*| (2^-8 for bf16, 2^-11 for fp16).
"""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s

from gpu_helpers import assert_close, device, ensure_built, upload_graph

pytestmark = pytest.mark.gpu

U16 = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    ensure_built()


def _rand(shape, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return graphgen.to_dtype((rng.standard_normal(shape) * scale).astype(np.float32), dtype)


def _check_projection(Y, X, W, dtype, out_dtype, rows=None):
    if rows is not None:
        X = X[torch.from_numpy(np.asarray(rows))]
    x, w = oracle.decode(dtype, X), oracle.decode(dtype, W)
    want = x @ w.T
    kin = x.shape[1]
    gamma = kin * 2.0 ** -24 / (1 - kin * 2.0 ** -24)
    bound = 2 * gamma * (np.abs(x) @ np.abs(w).T) + 1e-30
    if out_dtype != "f32":
        bound = bound + U16[out_dtype] * np.abs(want)
    got = Y.double().cpu().numpy()
    excess = np.abs(got - want) - bound
    assert excess.max() <= 0, "projection error exceeds its bound by %.3g" % excess.max()


SHAPES = [(1000, 128, 384, 128), (777, 64, 192, 64), (1, 8, 64, 64), (300, 200, 128, 128), (129, 512, 1536, 512),
          (5000, 128, 128, 128), (333, 96, 128, 64)]


@pytest.mark.parametrize("M,Kin,Nout,seg", SHAPES, ids=["%dx%dx%d/%d" % s for s in SHAPES])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("out", ["same", "f32"])
def test_linear_matches_oracle(M, Kin, Nout, seg, dtype, out):
    dev = device()
    X = _rand((M, Kin), dtype, 1)
    W = _rand((Nout, Kin), dtype, 2, scale=Kin ** -0.5)
    odt = dtype if out == "same" else "f32"
    Ys = g3s.linear(X.to(dev), W.to(dev), seg_cols=seg, out_dtype=odt)
    torch.cuda.synchronize()
    assert len(Ys) == Nout // seg
    _check_projection(torch.cat(Ys, dim=1), X, W, dtype, odt)


def test_linear_argument_errors():
    dev = device()
    X = _rand((64, 24), "bf16", 3).to(dev)
    W = _rand((64, 24), "bf16", 4).to(dev)
    with pytest.raises(g3s.G3SError):
        g3s.linear(X[:, :20].contiguous(), W[:, :20].contiguous())  # Kin not a multiple of 8
    with pytest.raises(g3s.G3SError):
        g3s.linear(X, _rand((96, 24), "bf16", 5).to(dev), seg_cols=32)  # segment not a multiple of 64
    with pytest.raises(g3s.G3SError):
        g3s.linear(X, _rand((256, 24), "bf16", 6).to(dev), seg_cols=64)  # four segments


def test_linear_full_size_sampled_rows():
    """The projection of the large workload's node features: 2M rows, Kin = 128,
    Q|K|V of 4 x 32 each; checked on sampled rows and both ends."""
    dev = device()
    M, kin, hd = 2_000_000, 128, 128
    X = _rand((M, kin), "bf16", 9).to(dev)
    W = _rand((3 * hd, kin), "bf16", 10, scale=kin ** -0.5).to(dev)
    Ys = g3s.linear(X, W, seg_cols=hd)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(11).choice(M, 4000, replace=False), [0, 1, M - 1]]))
    sel = torch.from_numpy(rows).to(dev)
    got = torch.cat([y[sel] for y in Ys], dim=1)
    _check_projection(got, X.cpu(), W.cpu(), "bf16", "bf16", rows=rows)


def _layer_case(g, H, d, dtype, variant, kin, ke=0, seed=20):
    dev = device()
    rp, ci = upload_graph(g)
    plan = g3s.Plan(rp, ci, g.num_nodes, H, d, dtype, variant)
    hd = H * d
    X = _rand((g.num_nodes, kin), dtype, seed)
    W = _rand((3 * hd, kin), dtype, seed + 1, scale=kin ** -0.5)
    Xe = We = None
    if variant == "rtmscore":
        Xe = _rand((g.num_edges, ke), dtype, seed + 2)
        We = _rand((hd, ke), dtype, seed + 3, scale=ke ** -0.5)
    out, (Q, K, V, E) = plan.layer_forward(X.to(dev), W.to(dev), None if Xe is None else Xe.to(dev),
                                           None if We is None else We.to(dev), want_eout=variant == "rtmscore")
    torch.cuda.synchronize()
    # the oracle: fp64 projections stored in the input type, then the attention definition
    proj = oracle.round_to(oracle.linear(X, W, dtype), dtype)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    qs, ks, vs = (torch.from_numpy(proj[:, i * hd:(i + 1) * hd].reshape(-1, H, d)).to(tdt) for i in range(3))
    es = None
    if variant == "rtmscore":
        es = torch.from_numpy(oracle.round_to(oracle.linear(Xe, We, dtype), dtype).reshape(-1, H, d)).to(tdt)
    # the GPU's stored projections agree with the rounded fp64 ones to the projection bound
    _check_projection(torch.cat([t.reshape(g.num_nodes, hd) for t in (Q, K, V)], dim=1), X, W, dtype, dtype)
    res = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, H, d, dtype, variant, qs, ks, vs, es,
                         want_eout=variant == "rtmscore")
    if variant == "rtmscore":
        O, Eout = out
        assert_close(O, res[0], dtype, "O")
        assert_close(Eout, res[1], dtype, "Eout")
    else:
        assert_close(out, res, dtype, "O")


def test_layer_standard_lognormal():
    g = graphgen.lognormal_local(num_nodes=3000, radius=128, seed=31)
    _layer_case(g, 4, 32, "bf16", "standard", kin=128)


def test_layer_standard_fp16_batched():
    g = graphgen.batched_dense(num_graphs=20, seed=32)
    _layer_case(g, 2, 64, "f16", "standard", kin=96)


def test_layer_rtmscore():
    g = graphgen.rtmscore_batch(num_graphs=4, min_nodes=30, max_nodes=60, seed=33)
    _layer_case(g, 8, 16, "bf16", "rtmscore", kin=128, ke=64)
