"""Python binding of libg3s (fused sparse graph attention on GB300).

Argument marshalling only: torch tensors are turned into raw device pointers
and a stream handle, and every step runs in the CUDA library through its C
ABI (``include/g3s.h``).  PyTorch provides device memory and streams.  There
is no CPU fallback: when ``libg3s.so`` is missing, importing works but every
call raises ``RuntimeError``.

    plan = Plan(row_ptr, col_idx, num_nodes, heads, head_dim, "bf16")
    O = plan.forward(Q, K, V)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libg3s.so")

G3S_OK = 0
STATUS_NAMES = {0: "G3S_OK", 1: "G3S_ERR_INVALID_ARG", 2: "G3S_ERR_UNSUPPORTED", 3: "G3S_ERR_BAD_GRAPH",
                4: "G3S_ERR_WORKSPACE", 5: "G3S_ERR_CUDA", 6: "G3S_ERR_TIMEOUT"}
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
VARIANTS = {"standard": 0, "rtmscore": 1}
NUM_BUCKETS = 5
ARRAYS = {  # name -> (enum, numpy dtype, trailing shape)
    "bucket_ptr": (0, np.int32, ()),
    "bucket_rows": (1, np.int32, ()),
    "heavy_rows": (2, np.int32, ()),
    "heavy_chunk_ptr": (3, np.int32, ()),
    "chunks": (4, np.int32, (3,)),
    "win_tile_ptr": (5, np.int32, ()),
    "tile_cols": (6, np.int32, ()),
    "tile_bits": (7, np.uint32, (4,)),
    "win_nnz": (8, np.int32, ()),
    "win_flags": (9, np.uint8, ()),
    "tile_windows": (10, np.int32, ()),
    "core_windows": (11, np.int32, ()),
    "tile_items": (12, np.int32, (8,)),
    "merge_rows": (13, np.int32, ()),
    "merge_ranges": (14, np.int32, (2,)),
}


class G3SError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class PlanOptions(ctypes.Structure):
    _fields_ = [
        ("bucket_bounds", ctypes.c_int32 * (NUM_BUCKETS - 2)),
        ("heavy_threshold", ctypes.c_int32),
        ("chunk_edges", ctypes.c_int32),
        ("bsb", ctypes.c_int32),
        ("tile_path", ctypes.c_int32),
        ("tile_density_milli", ctypes.c_int32),
        ("tile_max_tiles", ctypes.c_int32),
        ("bsb_smem_edges", ctypes.c_int32),
        ("rtm_elementwise_clamp", ctypes.c_int32),
        ("rtm_epsilon", ctypes.c_float),
        ("validate_graph", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("pack_rows", ctypes.c_int32),
        ("tile_pool_density_milli", ctypes.c_int32),
        ("degree_buckets", ctypes.c_int32),
        ("small_graph_rows", ctypes.c_int32),
        ("tile_split_density_milli", ctypes.c_int32),
        ("tile_split_parallel", ctypes.c_int32),
    ]


class PlanStats(ctypes.Structure):
    _fields_ = [
        ("num_nodes", ctypes.c_int64), ("num_edges", ctypes.c_int64),
        ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("variant", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("bucket_count", ctypes.c_int64 * NUM_BUCKETS),
        ("heavy_rows", ctypes.c_int64), ("chunks", ctypes.c_int64),
        ("has_bsb", ctypes.c_int32), ("tile_path", ctypes.c_int32),
        ("windows", ctypes.c_int64), ("tiles", ctypes.c_int64), ("tile_windows", ctypes.c_int64),
        ("dup_windows", ctypes.c_int64), ("large_windows", ctypes.c_int64),
        ("tile_window_nnz", ctypes.c_int64),
        ("pack_rows", ctypes.c_int32), ("pack_limit", ctypes.c_int32),
        ("heavy_threshold", ctypes.c_int32), ("chunk_edges", ctypes.c_int32), ("short_rows", ctypes.c_int64),
        ("workspace_used", ctypes.c_size_t),
        ("tile_items", ctypes.c_int64),
        ("small_graph", ctypes.c_int32),
        ("split_windows", ctypes.c_int64),
        ("split_items", ctypes.c_int64),
        ("merge_rows", ctypes.c_int64),
    ]


_lock = threading.Lock()
_lib = None

EXPORTED = ["g3s_version", "g3s_status_string", "g3s_last_error", "g3s_plan_options_init",
            "g3s_plan_workspace_size", "g3s_plan_create", "g3s_plan_get_stats", "g3s_plan_export",
            "g3s_forward", "g3s_host_staging_size", "g3s_forward_host", "g3s_plan_destroy",
            "g3s_forward_noalloc", "g3s_forward_check", "g3s_aggregate", "g3s_selftest_wait_timeout",
            "g3s_plan_set_edge_ids", "g3s_linear", "g3s_layer_forward", "g3s_gather_probe"]
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def load_library(path: str = LIB_PATH):
    """Load and bind libg3s.so (raises RuntimeError when it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("libg3s.so is not built (%s); run `python -m sparse_graph_attention_gb300.build` "
                               "or __graft_entry__.build()" % path)
        lib = ctypes.CDLL(path)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.g3s_version.restype = ctypes.c_char_p
        lib.g3s_status_string.argtypes = [I]
        lib.g3s_status_string.restype = ctypes.c_char_p
        lib.g3s_last_error.restype = ctypes.c_char_p
        lib.g3s_plan_options_init.argtypes = [ctypes.POINTER(PlanOptions)]
        lib.g3s_plan_options_init.restype = None
        lib.g3s_plan_workspace_size.argtypes = [I64, I64, I, I, I, I, ctypes.POINTER(PlanOptions),
                                                ctypes.POINTER(SZ)]
        lib.g3s_plan_create.argtypes = [P, P, I64, I64, I, I, I, I, ctypes.POINTER(PlanOptions), P, SZ, P,
                                        ctypes.POINTER(P)]
        lib.g3s_plan_get_stats.argtypes = [P, ctypes.POINTER(PlanStats)]
        lib.g3s_plan_export.argtypes = [P, I, P, SZ, ctypes.POINTER(SZ)]
        lib.g3s_forward.argtypes = [P, P, P, P, P, P, P, P]
        lib.g3s_host_staging_size.argtypes = [P, ctypes.POINTER(SZ)]
        lib.g3s_forward_host.argtypes = [P, P, P, P, P, P, P, P, SZ, P]
        lib.g3s_plan_destroy.argtypes = [P]
        lib.g3s_plan_destroy.restype = None
        lib.g3s_forward_noalloc.argtypes = [P, P, I64, I64, I, I, I, I, P, P, P, P, P, P, P]
        lib.g3s_forward_noalloc.restype = I
        lib.g3s_forward_check.argtypes = [P, P]
        lib.g3s_forward_check.restype = I
        lib.g3s_aggregate.argtypes = [P, P, P, P, I, ctypes.c_float, P]
        lib.g3s_aggregate.restype = I
        lib.g3s_selftest_wait_timeout.argtypes = [P, ctypes.c_uint64, P]
        lib.g3s_selftest_wait_timeout.restype = I
        lib.g3s_plan_set_edge_ids.argtypes = [P, P, I64, P]
        lib.g3s_plan_set_edge_ids.restype = I
        lib.g3s_linear.argtypes = [P, P, I64, I, I, I, ctypes.POINTER(P), I, I, P, P]
        lib.g3s_linear.restype = I
        lib.g3s_layer_forward.argtypes = [P, P, P, I, P, P, I, P, P, P, P, P, P, P]
        lib.g3s_layer_forward.restype = I
        lib.g3s_gather_probe.argtypes = [P, I64, I, I64, I, I, P, ctypes.POINTER(I64), P]
        lib.g3s_gather_probe.restype = I
        for name in ("g3s_plan_workspace_size", "g3s_plan_create", "g3s_plan_get_stats", "g3s_plan_export",
                     "g3s_forward", "g3s_host_staging_size", "g3s_forward_host"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def _check(status: int):
    if status != G3S_OK:
        raise G3SError(status, load_library().g3s_last_error().decode())


def version() -> str:
    return load_library().g3s_version().decode()


def default_options() -> PlanOptions:
    o = PlanOptions()
    load_library().g3s_plan_options_init(ctypes.byref(o))
    return o


def make_options(**kw) -> PlanOptions:
    o = default_options()
    for k, v in kw.items():
        if k == "bucket_bounds":
            for i, b in enumerate(v):
                o.bucket_bounds[i] = int(b)
        elif k == "bsb" or k == "tile_path" or k == "validate_graph" or k == "rtm_elementwise_clamp":
            setattr(o, k, int(v) if not isinstance(v, bool) else (1 if v else 0))
        elif k == "rtm_epsilon":
            o.rtm_epsilon = float(v)
        elif k == "out_dtype":
            o.out_dtype = DTYPES[v] if isinstance(v, str) else int(v)
        elif hasattr(o, k):
            setattr(o, k, int(v))
        else:
            raise TypeError("unknown plan option %r" % k)
    return o


def workspace_size(num_nodes, num_edges, heads, head_dim, dtype, variant="standard", **options) -> int:
    lib = load_library()
    n = ctypes.c_size_t()
    o = make_options(**options)
    _check(lib.g3s_plan_workspace_size(int(num_nodes), int(num_edges), int(heads), int(head_dim), DTYPES[dtype],
                                       VARIANTS[variant], ctypes.byref(o), ctypes.byref(n)))
    return int(n.value)


def _torch():
    import torch

    return torch


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


_TORCH_DTYPES = None


def torch_dtype(dtype: str):
    torch = _torch()
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def _dev_ptr(t, name, dtype=None, numel=None, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if numel is not None and t.numel() != numel:
        raise ValueError("%s has %d elements, expected %d" % (name, t.numel(), numel))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    return t.data_ptr()


def _host_ptr(t, name, dtype=None, numel=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CPU tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if numel is not None and t.numel() != numel:
        raise ValueError("%s has %d elements, expected %d" % (name, t.numel(), numel))
    return t.data_ptr()


class Plan:
    """A g3s plan for one graph (``g3s_plan_create`` / ``g3s_plan_destroy``).

    ``row_ptr`` and ``col_idx`` are int32 CUDA tensors; the plan keeps
    references to them and to its workspace, which torch allocates.
    """

    def __init__(self, row_ptr, col_idx, num_nodes: int, heads: int, head_dim: int, dtype: str = "f32",
                 variant: str = "standard", stream=None, **options):
        torch = _torch()
        lib = load_library()
        self._lib = lib
        self._handle = None
        self.num_nodes = int(num_nodes)
        self.num_edges = int(col_idx.numel())
        self.heads, self.head_dim, self.dtype, self.variant = int(heads), int(head_dim), dtype, variant
        self.device = row_ptr.device
        rp = _dev_ptr(row_ptr, "row_ptr", torch.int32, self.num_nodes + 1)
        ci = _dev_ptr(col_idx, "col_idx", torch.int32, device=self.device) if self.num_edges else 0
        self.options = make_options(**options)
        self.out_dtype = {v: k for k, v in DTYPES.items()}[self.options.out_dtype]
        n = ctypes.c_size_t()
        _check(lib.g3s_plan_workspace_size(self.num_nodes, self.num_edges, self.heads, self.head_dim, DTYPES[dtype],
                                           VARIANTS[variant], ctypes.byref(self.options), ctypes.byref(n)))
        self.workspace = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(lib.g3s_plan_create(rp, ci or None, self.num_nodes, self.num_edges, self.heads, self.head_dim,
                                       DTYPES[dtype], VARIANTS[variant], ctypes.byref(self.options),
                                       self.workspace.data_ptr(), self.workspace.numel(), _stream_handle(stream),
                                       ctypes.byref(h)))
        self._handle = h
        self.row_ptr, self.col_idx = row_ptr, col_idx
        self.edge_slots = self.num_edges
        self.edge_id = None

    def set_edge_ids(self, edge_id, num_edge_slots: int, stream=None):
        """``g3s_plan_set_edge_ids``: CSR position -> physical edge slot (None to clear)."""
        torch = _torch()
        ptr = _dev_ptr(edge_id, "edge_id", torch.int32, self.num_edges, self.device) if edge_id is not None else None
        with torch.cuda.device(self.device):
            _check(self._lib.g3s_plan_set_edge_ids(self.handle, ptr, int(num_edge_slots) if edge_id is not None else 0,
                                                   _stream_handle(stream)))
        self.edge_id = edge_id
        self.edge_slots = int(num_edge_slots) if edge_id is not None else self.num_edges

    # -- lifetime -----------------------------------------------------------
    def close(self):
        if self._handle is not None and self._handle.value:
            self._lib.g3s_plan_destroy(self._handle)
        self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        if self._handle is None:
            raise RuntimeError("plan is closed")
        return self._handle

    # -- introspection ------------------------------------------------------
    def stats(self) -> dict:
        s = PlanStats()
        _check(self._lib.g3s_plan_get_stats(self.handle, ctypes.byref(s)))
        out = {k: getattr(s, k) for k, _ in PlanStats._fields_}
        out["bucket_count"] = list(s.bucket_count)
        return out

    def export(self, name: str) -> np.ndarray:
        enum, dt, tail = ARRAYS[name]
        need = ctypes.c_size_t()
        _check(self._lib.g3s_plan_export(self.handle, enum, None, 0, ctypes.byref(need)))
        out = np.empty(need.value // np.dtype(dt).itemsize, dtype=dt)
        if need.value:
            _check(self._lib.g3s_plan_export(self.handle, enum, out.ctypes.data, need.value, ctypes.byref(need)))
        return out.reshape((-1,) + tail) if tail else out

    # -- compute ------------------------------------------------------------
    def _node_numel(self):
        return self.num_nodes * self.heads * self.head_dim

    def forward(self, Q, K, V, E=None, O=None, Eout=None, want_eout: bool = False, stream=None):
        """``g3s_forward``: returns O, or (O, Eout) when ``want_eout`` (RTMScore)."""
        torch = _torch()
        tdt = torch_dtype(self.dtype)
        odt = torch_dtype(self.out_dtype)
        nn = self._node_numel()
        ne = self.edge_slots * self.heads * self.head_dim
        q = _dev_ptr(Q, "Q", tdt, nn, self.device)
        k = _dev_ptr(K, "K", tdt, nn, self.device)
        v = _dev_ptr(V, "V", tdt, nn, self.device)
        if O is None:
            O = torch.empty((self.num_nodes, self.heads, self.head_dim), dtype=odt, device=self.device)
        o = _dev_ptr(O, "O", odt, nn, self.device)
        e = eo = None
        if self.variant == "rtmscore":
            e = _dev_ptr(E, "E", tdt, ne, self.device) if self.num_edges else None
            if want_eout and Eout is None:
                Eout = torch.empty((self.edge_slots, self.heads, self.head_dim), dtype=odt, device=self.device)
            if Eout is not None:
                eo = _dev_ptr(Eout, "Eout", odt, ne, self.device)
        elif E is not None or Eout is not None:
            raise ValueError("E / Eout are only valid for an RTMScore plan")
        with torch.cuda.device(self.device):
            _check(self._lib.g3s_forward(self.handle, q, k, v, e, o, eo, _stream_handle(stream)))
        return (O, Eout) if want_eout else O

    def layer_forward(self, X, Wqkv, Xe=None, We=None, O=None, Eout=None, want_eout: bool = False,
                      stream=None):
        """``g3s_layer_forward``: Q|K|V = X Wqkv^T (and, for RTMScore, Eproj = Xe We^T),
        then the fused forward.  Returns (O, (Q, K, V, Eproj)) or, with
        ``want_eout``, ((O, Eout), (Q, K, V, Eproj))."""
        torch = _torch()
        tdt = torch_dtype(self.dtype)
        odt = torch_dtype(self.out_dtype)
        hd = self.heads * self.head_dim
        kin = int(X.shape[-1])
        x = _dev_ptr(X, "X", tdt, self.num_nodes * kin, self.device)
        wqkv = _dev_ptr(Wqkv, "Wqkv", tdt, 3 * hd * kin, self.device)
        Q, K, V = (torch.empty((self.num_nodes, self.heads, self.head_dim), dtype=tdt, device=self.device)
                   for _ in range(3))
        E = xe = we = ep = None
        ke = 0
        if self.variant == "rtmscore":
            ke = int(Xe.shape[-1])
            xe = _dev_ptr(Xe, "Xe", tdt, self.edge_slots * ke, self.device)
            we = _dev_ptr(We, "We", tdt, hd * ke, self.device)
            E = torch.empty((self.edge_slots, self.heads, self.head_dim), dtype=tdt, device=self.device)
            ep = E.data_ptr()
            if want_eout and Eout is None:
                Eout = torch.empty((self.edge_slots, self.heads, self.head_dim), dtype=odt, device=self.device)
        elif Xe is not None or We is not None:
            raise ValueError("Xe / We are only valid for an RTMScore plan")
        if O is None:
            O = torch.empty((self.num_nodes, self.heads, self.head_dim), dtype=odt, device=self.device)
        o = _dev_ptr(O, "O", odt, self._node_numel(), self.device)
        eo = Eout.data_ptr() if Eout is not None else None
        with torch.cuda.device(self.device):
            _check(self._lib.g3s_layer_forward(self.handle, x, wqkv, kin, xe, we, ke, Q.data_ptr(), K.data_ptr(),
                                               V.data_ptr(), ep, o, eo, _stream_handle(stream)))
        out = (O, Eout) if want_eout else O
        return out, (Q, K, V, E)

    def aggregate(self, W, X, O=None, normalize: bool = False, eps: float = 1e-6, stream=None):
        """``g3s_aggregate``: O_i = sum_e W[e] X[src(e)] (optionally / (sum_e W[e] + eps))."""
        torch = _torch()
        tdt = torch_dtype(self.dtype)
        odt = torch_dtype(self.out_dtype)
        nn = self._node_numel()
        w = _dev_ptr(W, "W", tdt, self.edge_slots * self.heads, self.device) if self.num_edges else None
        x = _dev_ptr(X, "X", tdt, nn, self.device)
        if O is None:
            O = torch.empty((self.num_nodes, self.heads, self.head_dim), dtype=odt, device=self.device)
        o = _dev_ptr(O, "O", odt, nn, self.device)
        with torch.cuda.device(self.device):
            _check(self._lib.g3s_aggregate(self.handle, w, x, o, 1 if normalize else 0, float(eps),
                                           _stream_handle(stream)))
        return O

    def check(self, stream=None):
        """``g3s_forward_check``: synchronise and raise G3SError(G3S_ERR_TIMEOUT)
        if a forward kernel gave up a bounded device wait."""
        _check(self._lib.g3s_forward_check(self.handle, _stream_handle(stream)))

    def staging_size(self) -> int:
        n = ctypes.c_size_t()
        _check(self._lib.g3s_host_staging_size(self.handle, ctypes.byref(n)))
        return int(n.value)

    def forward_host(self, Qh, Kh, Vh, Oh, Eh=None, Eouth=None, staging=None, stream=None):
        """``g3s_forward_host``: host (ideally pinned) tensors in and out, device staging.

        Enqueued on ``stream``; synchronise before reading ``Oh``.
        """
        torch = _torch()
        tdt = torch_dtype(self.dtype)
        odt = torch_dtype(self.out_dtype)
        nn = self._node_numel()
        ne = self.edge_slots * self.heads * self.head_dim
        if staging is None:
            staging = torch.empty(self.staging_size(), dtype=torch.uint8, device=self.device)
        ptrs = [_host_ptr(Qh, "Q", tdt, nn), _host_ptr(Kh, "K", tdt, nn), _host_ptr(Vh, "V", tdt, nn)]
        e = _host_ptr(Eh, "E", tdt, ne) if Eh is not None else None
        o = _host_ptr(Oh, "O", odt, nn)
        eo = _host_ptr(Eouth, "Eout", odt, ne) if Eouth is not None else None
        with torch.cuda.device(self.device):
            _check(self._lib.g3s_forward_host(self.handle, ptrs[0], ptrs[1], ptrs[2], e, o, eo,
                                              _dev_ptr(staging, "staging", torch.uint8, device=self.device),
                                              staging.numel(), _stream_handle(stream)))
        return staging


def linear(X, W, seg_cols: Optional[int] = None, out_dtype: Optional[str] = None, outs=None, status=None,
           stream=None):
    """``g3s_linear``: Y = X W^T for X (M, Kin) and W (Nout, Kin), 16-bit, on
    the tensor cores.  Returns a list of Nout / seg_cols outputs of shape
    (M, seg_cols) (default seg_cols = Nout)."""
    torch = _torch()
    lib = load_library()
    names = {torch.float16: "f16", torch.bfloat16: "bf16"}
    if X.dtype not in names:
        raise TypeError("X must be fp16 or bf16")
    dt = names[X.dtype]
    M, kin = int(X.shape[0]), int(X.shape[-1])
    nout = int(W.shape[0])
    seg = int(seg_cols or nout)
    odt = out_dtype or dt
    if outs is None:
        outs = [torch.empty((M, seg), dtype=torch_dtype(odt), device=X.device) for _ in range(nout // seg)]
    ptrs = (ctypes.c_void_p * len(outs))(*[_dev_ptr(o, "Y", torch_dtype(odt), M * seg, X.device) for o in outs])
    st = _dev_ptr(status, "status", torch.int32, 1, X.device) if status is not None else None
    with torch.cuda.device(X.device):
        _check(lib.g3s_linear(_dev_ptr(X, "X", X.dtype, M * kin, X.device), _dev_ptr(W, "W", X.dtype, nout * kin,
                                                                                  X.device),
                              M, kin, nout, DTYPES[dt], ptrs, seg, DTYPES[odt], st, _stream_handle(stream)))
    return outs


def gather_probe(src, row_bytes: int, gathers: int, ctas: int, sink, plain_loads: bool = False, stream=None) -> int:
    """``g3s_gather_probe``: read ``gathers`` (rounded up) hashed random rows of
    ``row_bytes`` from the CUDA tensor ``src`` (a power-of-two number of rows);
    returns the rows read.  A measurement aid (no attention arithmetic): the
    rate at which the CUDA-core kernel's gathers can be served."""
    lib = load_library()
    nbytes = src.numel() * src.element_size()
    if nbytes % row_bytes:
        raise ValueError("src size must be a multiple of row_bytes")
    got = ctypes.c_int64()
    _check(lib.g3s_gather_probe(_dev_ptr(src, "src"), nbytes // row_bytes, int(row_bytes), int(gathers), int(ctas),
                                1 if plain_loads else 0, _dev_ptr(sink, "sink"), ctypes.byref(got),
                                _stream_handle(stream)))
    return got.value


def forward_noalloc(row_ptr, col_idx, num_nodes, heads, head_dim, dtype, variant, Q, K, V, E=None, O=None,
                    Eout=None, stream=None):
    """``g3s_forward_noalloc``: plan + forward in one call using the library's
    static device scratch (for callers that cannot allocate device memory).
    Returns O (fp32), and Eout when given."""
    torch = _torch()
    lib = load_library()
    dev = row_ptr.device
    n, ne = int(num_nodes), int(col_idx.numel())
    tdt = torch_dtype(dtype)
    nn, nedge = n * heads * head_dim, ne * heads * head_dim
    if O is None:
        O = torch.empty((n, heads, head_dim), dtype=torch.float32, device=dev)
    args = [_dev_ptr(row_ptr, "row_ptr", torch.int32, n + 1, dev),
            _dev_ptr(col_idx, "col_idx", torch.int32, device=dev) if ne else None]
    vals = [_dev_ptr(Q, "Q", tdt, nn, dev), _dev_ptr(K, "K", tdt, nn, dev), _dev_ptr(V, "V", tdt, nn, dev),
            _dev_ptr(E, "E", tdt, nedge, dev) if E is not None else None,
            _dev_ptr(O, "O", torch.float32, nn, dev),
            _dev_ptr(Eout, "Eout", torch.float32, nedge, dev) if Eout is not None else None]
    with torch.cuda.device(dev):
        _check(lib.g3s_forward_noalloc(args[0], args[1], n, ne, int(heads), int(head_dim), DTYPES[dtype],
                                       VARIANTS[variant], *vals, _stream_handle(stream)))
    return (O, Eout) if Eout is not None else O


__all__ = ["gather_probe", "forward_noalloc", "linear", "Plan", "G3SError", "load_library", "version", "workspace_size", "make_options", "default_options",
           "DTYPES", "VARIANTS", "ARRAYS", "EXPORTED", "LIB_PATH"]
