"""Shared helpers of the GPU tests: build inputs, run the library, compare
with the fp64 oracle under the tolerances of the contract:

* fp32 inputs:      max |O - O*| <= 1e-4 (and the same for Eout)
* fp16/bf16 inputs: max |O - O*| / max |O*| <= 3e-3 (same rule for Eout)

O is fp32 by default (the accumulation type).  When a plan stores O in the
16-bit input type, the store itself may add half an ulp: up to 2^-8 |O*| for
bf16 and 2^-11 |O*| for fp16 -- more than 3e-3 of the output scale for bf16
values just above a power of two -- so those outputs are checked elementwise
against 3e-3 max|O*| + u |O*| (``assert_close_stored16``).
"""
from __future__ import annotations

import numpy as np
import torch

import graphgen
import oracle
import sparse_graph_attention_gb300 as g3s
from sparse_graph_attention_gb300 import build as g3s_build

TOL_F32 = 1e-4
TOL_REL16 = 3e-3

_built = False


def ensure_built():
    global _built
    if not _built:
        g3s_build.build()
        g3s.load_library()
        _built = True


def device():
    return torch.device("cuda:0")


def upload_graph(g):
    dev = device()
    return (torch.from_numpy(g.row_ptr.astype(np.int32)).to(dev),
            torch.from_numpy(g.col_idx.astype(np.int32)).to(dev))


def cast_values(vals, dtype):
    """fp32 numpy values -> dict of CPU torch tensors in ``dtype`` (RNE)."""
    return {k: graphgen.to_dtype(v, dtype) for k, v in vals.items()}


def error(got, want, dtype):
    g = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert g.shape == want.shape, (g.shape, want.shape)
    if g.size == 0:
        return 0.0
    assert np.all(np.isfinite(g)), "non-finite output"
    diff = np.abs(g - want).max()
    if dtype == "f32":
        return float(diff)
    scale = np.abs(want).max()
    return float(diff / scale) if scale > 0 else float(diff)


def assert_close(got, want, dtype, what="O"):
    err = error(got, want, dtype)
    tol = TOL_F32 if dtype == "f32" else TOL_REL16
    assert err <= tol, "%s error %.3g > %.3g (%s)" % (what, err, tol, dtype)
    return err


UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def assert_close_stored16(got, want, dtype, what="O"):
    g = got.detach().double().cpu().numpy()
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(g))
    bound = TOL_REL16 * np.abs(want).max() + UNIT_ROUNDOFF[dtype] * np.abs(want)
    excess = np.abs(g - want) - bound
    assert excess.max() <= 0, "%s exceeds 3e-3*max|O*| + u|O*| by %.3g" % (what, excess.max())
    return float(np.abs(g - want).max() / max(np.abs(want).max(), 1e-30))


def run_case(g, vals, heads, head_dim, dtype, variant, rows=None, check_eout=True, plan_kw=None,
             oracle_kw=None):
    """Plan + forward on the GPU, oracle on ``rows`` (default all); asserts and returns errors."""
    ensure_built()
    plan_kw = dict(plan_kw or {})
    oracle_kw = dict(oracle_kw or {})
    if variant == "rtmscore":
        plan_kw.setdefault("rtm_elementwise_clamp", oracle_kw.get("elementwise_clamp", True))
    dev = device()
    rp, ci = upload_graph(g)
    t = cast_values(vals, dtype)
    plan = g3s.Plan(rp, ci, g.num_nodes, heads, head_dim, dtype, variant, **plan_kw)
    Q, K, V = (t[k].to(dev) for k in ("Q", "K", "V"))
    E = t["E"].to(dev) if variant == "rtmscore" else None
    if variant == "rtmscore":
        O, Eout = plan.forward(Q, K, V, E, want_eout=True)
    else:
        O = plan.forward(Q, K, V)
    torch.cuda.synchronize()
    sel = np.arange(g.num_nodes) if rows is None else np.asarray(rows)
    res = oracle.forward(g.row_ptr, g.col_idx, g.num_nodes, heads, head_dim, dtype, variant, t["Q"], t["K"], t["V"],
                         t.get("E"), rows=sel, want_eout=(variant == "rtmscore" and check_eout), **oracle_kw)
    errs = {}
    if variant == "rtmscore" and check_eout:
        Ostar, Estar = res
    else:
        Ostar = res
    stored16 = plan.out_dtype != "f32"
    check = (lambda a, b, w: assert_close_stored16(a, b, dtype, w)) if stored16 else \
        (lambda a, b, w: assert_close(a, b, dtype, w))
    errs["O"] = check(O[torch.from_numpy(sel).to(dev)], Ostar, "O")
    if variant == "rtmscore" and check_eout:
        if rows is None:
            errs["Eout"] = check(Eout, Estar, "Eout")
        else:
            pos = np.concatenate([np.arange(g.row_ptr[r], g.row_ptr[r + 1]) for r in sel]).astype(np.int64)
            errs["Eout"] = check(Eout[torch.from_numpy(pos).to(dev)], Estar[pos], "Eout")
    return plan, O, errs
