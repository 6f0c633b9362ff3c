"""fp64 CPU oracle for fused sparse graph attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product library never loads it, and it never loads the product library.

* ``forward``   -- the attention definitions, in C (``g3s_oracle.c``), fp64,
                   OpenMP over rows.
* ``aggregate`` -- the weighted (optionally normalised) aggregation, same file.
* ``linear``    -- the projection Y = X W^T in fp64 (numpy matmul on the
                   exactly widened inputs), and ``round_to`` for storing a
                   projection in a 16-bit type (round to nearest even).
* ``decode``    -- the exact widening of stored fp32 / fp16 / bf16 values.
* ``planner``   -- numpy reference of the degree buckets, heavy-row chunks and
                   BSB tiles (``planner.py``).

Every function here is pinned by ``tests/test_oracle_pins.py`` and
``tests/test_planner_oracle.py`` to brute force, a hand-worked example,
closed forms and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import planner  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "g3s_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libg3s_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
VARIANTS = {"standard": 0, "rtmscore": 1}


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2 -fopenmp) into oracle/_build."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.g3s_oracle_forward.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, P, P, P, P, P,
                                       ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_double]
    lib.g3s_oracle_forward.restype = ctypes.c_int
    lib.g3s_oracle_decode.argtypes = [ctypes.c_int, P, ctypes.c_int64, P]
    lib.g3s_oracle_decode.restype = ctypes.c_int
    lib.g3s_oracle_threads.restype = ctypes.c_int
    lib.g3s_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.g3s_oracle_set_threads.restype = None
    lib.g3s_oracle_aggregate.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P,
                                         ctypes.c_int64, P, ctypes.c_int, ctypes.c_double]
    lib.g3s_oracle_aggregate.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def load_library(path: str):
    """Bind an oracle shared library at ``path`` (used to load planted-mistake copies in tests)."""
    return _bind(path)


def threads() -> int:
    return int(_load().g3s_oracle_threads())


def set_threads(n: int) -> None:
    """Threads the oracle's later calls use (results do not depend on it)."""
    _load().g3s_oracle_set_threads(int(n))


def _raw(x, dtype: str) -> np.ndarray:
    """Stored bytes of a value array: float32 for f32, the uint16 bit pattern otherwise.

    Accepts numpy arrays or torch CPU tensors (16-bit tensors are viewed as int16).
    """
    if x is None:
        return None
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if dtype == "f32":
                return np.ascontiguousarray(x.to(torch.float32).numpy())
            return np.ascontiguousarray(x.view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype == "f32":
        if x.dtype != np.float32:
            raise TypeError("f32 oracle input must be float32")
        return x
    if x.dtype == np.float16 and dtype == "f16":
        return x.view(np.uint16)
    if x.dtype not in (np.uint16, np.int16):
        raise TypeError("16-bit oracle input must be given as its uint16 bit pattern")
    return x.view(np.uint16)


def decode(dtype: str, bits) -> np.ndarray:
    raw = _raw(bits, dtype)
    out = np.empty(raw.size, np.float64)
    rc = _load().g3s_oracle_decode(DTYPES[dtype], raw.ctypes.data, raw.size, out.ctypes.data)
    if rc:
        raise ValueError("bad dtype")
    return out.reshape(raw.shape)


def forward(row_ptr, col_idx, num_nodes, heads, head_dim, dtype, variant, Q, K, V, E=None,
            rows=None, want_eout=False, elementwise_clamp=True, eps=1e-6, lib=None):
    """fp64 attention for ``rows`` (default: all rows).

    Returns ``O`` of shape (len(rows), H, d) and, when ``want_eout`` (RTMScore),
    ``Eout`` of shape (E, H, d) whose entries for edges of unlisted rows are NaN.
    """
    lib = lib if lib is not None else _load()
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = int(num_nodes)
    if rows is None:
        rows = np.arange(n, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    q, k, v = _raw(Q, dtype), _raw(K, dtype), _raw(V, dtype)
    e = _raw(E, dtype) if E is not None else None
    hd = heads * head_dim
    for name, a, cnt in (("Q", q, n), ("K", k, n), ("V", v, n)):
        if a.size != cnt * hd:
            raise ValueError("%s has %d elements, expected %d" % (name, a.size, cnt * hd))
    ne = int(col_idx.size)
    if variant == "rtmscore":
        if e is None or e.size != ne * hd:
            raise ValueError("RTMScore needs E of shape (E, H, d)")
    O = np.zeros((rows.size, heads, head_dim), np.float64)
    Eout = None
    if want_eout and variant == "rtmscore":
        Eout = np.full((ne, heads, head_dim), np.nan, np.float64)
    rc = lib.g3s_oracle_forward(row_ptr.ctypes.data, col_idx.ctypes.data, n, heads, head_dim,
                                DTYPES[dtype], VARIANTS[variant], q.ctypes.data, k.ctypes.data,
                                v.ctypes.data, e.ctypes.data if e is not None else None,
                                rows.ctypes.data, rows.size, O.ctypes.data,
                                Eout.ctypes.data if Eout is not None else None,
                                1 if elementwise_clamp else 0, float(eps))
    if rc == 2:
        raise ValueError("graph index out of range")
    if rc:
        raise ValueError("bad oracle arguments")
    return (O, Eout) if want_eout else O


def aggregate(row_ptr, col_idx, num_nodes, heads, head_dim, dtype, W, X, rows=None, normalize=False, eps=1e-6,
              lib=None):
    """fp64 weighted aggregation for ``rows`` (default all): O of shape (len(rows), H, d)."""
    lib = lib if lib is not None else _load()
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = int(num_nodes)
    rows = np.arange(n, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    w, x = _raw(W, dtype), _raw(X, dtype)
    if w.size != col_idx.size * heads:
        raise ValueError("W must have E*H elements")
    if x.size != n * heads * head_dim:
        raise ValueError("X must have N*H*d elements")
    O = np.zeros((rows.size, heads, head_dim), np.float64)
    rc = lib.g3s_oracle_aggregate(row_ptr.ctypes.data, col_idx.ctypes.data, n, heads, head_dim, DTYPES[dtype],
                                  w.ctypes.data, x.ctypes.data, rows.ctypes.data, rows.size, O.ctypes.data,
                                  1 if normalize else 0, float(eps))
    if rc == 2:
        raise ValueError("graph index out of range")
    if rc:
        raise ValueError("bad oracle arguments")
    return O


def linear(X, W, dtype: str) -> np.ndarray:
    """fp64 projection Y = X W^T of the stored values: X (M, Kin), W (Nout, Kin).

    The dense projection in front of the attention (the Triton article,
    stondelli.it/articles/gattn-triton, closing section: the GEMMs that remain
    once the attention is fused).  The inputs are widened exactly, the
    product is numpy's fp64 matmul."""
    x = decode(dtype, X)
    w = decode(dtype, W)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("need X (M, Kin) and W (Nout, Kin)")
    return x @ w.T


def round_to(y, dtype: str) -> np.ndarray:
    """Values of fp64 ``y`` once stored in ``dtype`` (round to nearest even), as fp64."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float64))
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return t.to(tdt).to(torch.float64).numpy()
