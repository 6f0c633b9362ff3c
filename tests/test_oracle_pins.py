"""The fp64 oracle against brute force, the worked example, closed forms and invariants."""
import numpy as np
import pytest
import torch

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
