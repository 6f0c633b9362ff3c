"""The fp64 oracle against brute force, the worked example, closed forms and invariants."""
import numpy as np
import pytest
import torch

import graphgen
import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.forward)


@pytest.mark.parametrize("pin", pins.AGG_PINS, ids=lambda p: p.__name__)
def test_aggregate_pin(pin):
    pin(oracle.aggregate)


def test_aggregate_sixteen_bit_inputs_read_exactly():
    import torch

    rp, col, q, k, v, _ = pins._graph_and_values(93)
    n, H, d = v.shape
    w = np.random.default_rng(1).standard_normal((col.size, H)).astype(np.float32)
    for tdt, name in ((torch.bfloat16, "bf16"), (torch.float16, "f16")):
        wt, xt = torch.from_numpy(w).to(tdt), torch.from_numpy(v).to(tdt)
        got = oracle.aggregate(rp, col, n, H, d, name, wt, xt, normalize=True)
        want = oracle.aggregate(rp, col, n, H, d, "f32", wt.float().numpy(), xt.float().numpy(), normalize=True)
        assert np.array_equal(got, want)


def test_decode_f16_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("f16", bits)
    want = bits.view(np.float16).astype(np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_decode_bf16_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("bf16", bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_row_subset_matches_full():
    rp, col, q, k, v, _ = pins._graph_and_values(81)
    n, H, d = q.shape
    full = oracle.forward(rp, col, n, H, d, "f32", "standard", q, k, v)
    rows = np.array([5, 0, n - 1, 17, 17])
    sub = oracle.forward(rp, col, n, H, d, "f32", "standard", q, k, v, rows=rows)
    assert np.array_equal(sub, full[rows])


def test_bad_index_is_reported():
    rp = np.array([0, 2, 3], np.int32)
    col = np.array([0, 5, 1], np.int32)
    x = np.zeros((2, 1, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.forward(rp, col, 2, 1, 4, "f32", "standard", x, x, x)


# ---------------------------------------------------------------------------
# the projection Y = X W^T and the 16-bit store
# ---------------------------------------------------------------------------
def test_linear_matches_brute_force():
    """oracle.linear against a triple loop on the widened values, rectangular
    and square (a transposed weight would fail the square case)."""
    rng = np.random.default_rng(7)
    for dt in ("bf16", "f16"):
        for (m, nout, kin) in ((5, 7, 12), (6, 6, 6)):
            X = graphgen.to_dtype(rng.standard_normal((m, kin)).astype(np.float32), dt)
            W = graphgen.to_dtype(rng.standard_normal((nout, kin)).astype(np.float32), dt)
            Y = oracle.linear(X, W, dt)
            x, w = oracle.decode(dt, X), oracle.decode(dt, W)
            for i in range(m):
                for j in range(nout):
                    acc = 0.0
                    for k in range(kin):
                        acc += x[i, k] * w[j, k]
                    assert abs(Y[i, j] - acc) <= 1e-12 * (1.0 + abs(acc))


def test_linear_selects_rows_of_w():
    """W with one 1 per row picks columns of X exactly (Y[:, j] = X[:, perm[j]])."""
    rng = np.random.default_rng(8)
    kin, nout = 16, 10
    perm = rng.integers(0, kin, nout)
    Wn = np.zeros((nout, kin), np.float32)
    Wn[np.arange(nout), perm] = 1.0
    X = graphgen.to_dtype(rng.standard_normal((9, kin)).astype(np.float32), "bf16")
    Y = oracle.linear(X, graphgen.to_dtype(Wn, "bf16"), "bf16")
    assert np.array_equal(Y, oracle.decode("bf16", X)[:, perm])


def test_round_to_ties_and_ranges():
    """Round to nearest even at the bf16 / fp16 half-ulp points."""
    one = 1.0
    assert oracle.round_to(np.array([one + 2.0 ** -8]), "bf16")[0] == 1.0          # tie -> even
    assert oracle.round_to(np.array([one + 3 * 2.0 ** -9]), "bf16")[0] == one + 2.0 ** -7
    assert oracle.round_to(np.array([one + 2.0 ** -11]), "f16")[0] == 1.0          # tie -> even
    assert oracle.round_to(np.array([one + 3 * 2.0 ** -12]), "f16")[0] == one + 2.0 ** -10
    assert oracle.round_to(np.array([-2.5]), "bf16")[0] == -2.5


def test_thread_count_does_not_change_results():
    """Each row is summed in a fixed order by one thread, so one thread and
    every thread give identical bits (the benchmark times both)."""
    g = graphgen.powerlaw(num_nodes=3000, max_degree=1500, seed=91)
    vals = graphgen.make_values(g.num_nodes, g.num_edges, 2, 32, True, seed=92)
    t = {k: graphgen.to_dtype(v, "bf16") for k, v in vals.items()}
    n_all = oracle.threads()
    outs = []
    for n in (1, n_all):
        oracle.set_threads(n)
        outs.append(oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, 2, 32, "bf16", "rtmscore", t["Q"], t["K"],
                                   t["V"], t["E"], want_eout=True))
    oracle.set_threads(n_all)
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1], equal_nan=True)
