"""Thin Python binding of the C ABI in ``include/gattn.h`` (ctypes).

Argument marshalling only: every step of the attention path runs in the CUDA
library ``_build/libgattn.so``.  There is no fallback -- if the library is not
built or cannot be loaded, every call raises.  PyTorch supplies device memory
and the current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

GATTN_OK = 0
STATUS = {0: "GATTN_OK", 1: "GATTN_ERR_INVALID_ARG", 2: "GATTN_ERR_BAD_GRAPH",
          3: "GATTN_ERR_UNSUPPORTED", 4: "GATTN_ERR_OOM", 5: "GATTN_ERR_CUDA",
          6: "GATTN_ERR_TIMEOUT"}
GATTN_F32, GATTN_BF16 = 0, 1
GATTN_SCORE_DOT, GATTN_SCORE_GATV2 = 0, 1
EXPORTED = ("gattn_plan_create", "gattn_plan_destroy", "gattn_plan_get_info",
            "gattn_plan_export", "gattn_workspace_size", "gattn_fwd", "gattn_bwd",
            "gattn_bwd_dq", "gattn_bwd_dkdv", "gattn_plan_check_errors", "gattn_fwd_noalloc",
            "gattn_plan_export_tiles", "gattn_plan_export_tile_bwd", "gattn_reorder", "gattn_permute_csr",
            "gattn_permute_rows", "gattn_pool_workspace_size", "gattn_pool_fwd",
            "gattn_pool_bwd", "gattn_spmm_workspace_size", "gattn_spmm",
            "gattn_plan_set_wait_test", "gattn_last_error", "gattn_version")


class GattnError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


class _Score(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("scale", ctypes.c_float), ("a", ctypes.c_void_p),
                ("neg_slope", ctypes.c_float)]


class _PlanOpts(ctypes.Structure):
    _fields_ = [("heavy_threshold", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("tile_enable", ctypes.c_int32), ("tile_density", ctypes.c_float)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("M", ctypes.c_int64),
                ("heavy_threshold", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("n_light", ctypes.c_int64), ("n_heavy", ctypes.c_int64),
                ("n_chunks", ctypes.c_int64), ("n_light_src", ctypes.c_int64),
                ("n_heavy_src", ctypes.c_int64), ("n_src_chunks", ctypes.c_int64),
                ("max_deg", ctypes.c_int32), ("max_outdeg", ctypes.c_int32),
                ("device_bytes", ctypes.c_size_t), ("n_tiles", ctypes.c_int64),
                ("n_tile_rows", ctypes.c_int64), ("tile_edges", ctypes.c_int64),
                ("tile_min_edges", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(path: str | None = None):
    """Load the CUDA library (no compute call is made).

    Without ``path`` the in-tree build is loaded once and cached for every
    call of this module.  With ``path`` that library is loaded and returned
    but not cached: the module's own calls keep using the default library
    unless the caller assigns the result to ``binding._lib``.
    """
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"gattn CUDA library not found at {p}; build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        st = ctypes.c_int
        lib.gattn_plan_create.argtypes = [P, P, i32, i64, ctypes.POINTER(_PlanOpts), P,
                                          ctypes.POINTER(P)]
        lib.gattn_plan_destroy.argtypes = [P]
        lib.gattn_plan_get_info.argtypes = [P, ctypes.POINTER(_PlanInfo)]
        lib.gattn_plan_export.argtypes = [P] + [P] * 11
        lib.gattn_workspace_size.argtypes = [P, i32, i32, ctypes.c_int, ctypes.POINTER(sz)]
        lib.gattn_fwd.argtypes = [P, i32, i32, ctypes.c_int, P, P, P, ctypes.POINTER(_Score), P,
                                  P, P, sz, P]
        lib.gattn_bwd.argtypes = [P, i32, i32, ctypes.c_int, P, P, P, ctypes.POINTER(_Score), P,
                                  P, P, P, P, P, P, P, sz, P]
        lib.gattn_bwd_dq.argtypes = [P, i32, i32, ctypes.c_int, P, P, P, ctypes.POINTER(_Score),
                                     P, P, P, P, P, P, sz, P]
        lib.gattn_bwd_dkdv.argtypes = [P, i32, i32, ctypes.c_int, P, P, P,
                                       ctypes.POINTER(_Score), P, P, P, P, P, sz, P]
        lib.gattn_plan_check_errors.argtypes = [P]
        lib.gattn_fwd_noalloc.argtypes = [P, i32, i32, ctypes.c_int, P, P, P,
                                          ctypes.POINTER(_Score), P, P, P]
        lib.gattn_plan_export_tiles.argtypes = [P] * 6
        lib.gattn_plan_export_tile_bwd.argtypes = [P, ctypes.POINTER(i64)] + [P] * 6
        lib.gattn_reorder.argtypes = [P, P, i32, i64, i32, P]
        lib.gattn_permute_csr.argtypes = [P, P, i32, i64, P, P, P]
        lib.gattn_permute_rows.argtypes = [P, P, P, i32, i64, i32, P]
        lib.gattn_pool_workspace_size.argtypes = [P, i32, ctypes.c_int, ctypes.POINTER(sz)]
        lib.gattn_pool_fwd.argtypes = [P, i32, ctypes.c_int, i32, P, P, P, P, sz, P]
        lib.gattn_pool_bwd.argtypes = [P, i32, ctypes.c_int, P, P, P, P, sz, P]
        lib.gattn_spmm_workspace_size.argtypes = [P, i32, ctypes.c_int, ctypes.POINTER(sz)]
        lib.gattn_spmm.argtypes = [P, i32, ctypes.c_int, P, P, P, i32, P, sz, P]
        lib.gattn_plan_set_wait_test.argtypes = [P, i32]
        for name in EXPORTED[:22]:
            getattr(lib, name).restype = st
        lib.gattn_last_error.restype = ctypes.c_char_p
        lib.gattn_last_error.argtypes = []
        lib.gattn_version.restype = ctypes.c_char_p
        lib.gattn_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def _check(status: int, where: str):
    if status != GATTN_OK:
        raise GattnError(status, where, load_library().gattn_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return GATTN_F32
    if dt == torch.bfloat16:
        return GATTN_BF16
    raise GattnError(1, "dtype", f"unsupported dtype {dt}")


class Score:
    """Score function: ``Score("dot", scale=0.0)`` or ``Score("gatv2", a=a, neg_slope=0.2)``.

    ``a`` is a CUDA fp32 tensor [H, D]; scale 0 means 1/sqrt(D).
    """

    def __init__(self, kind: str = "dot", scale: float = 0.0, a: torch.Tensor | None = None,
                 neg_slope: float = 0.2):
        if kind not in ("dot", "gatv2"):
            raise ValueError(kind)
        self.kind, self.scale, self.a, self.neg_slope = kind, scale, a, neg_slope

    def _struct(self):
        a = None
        if self.kind == "gatv2":
            if self.a is None or self.a.dtype != torch.float32 or not self.a.is_contiguous():
                raise ValueError("GATv2 needs a contiguous fp32 CUDA tensor a[H, D]")
            a = self.a.data_ptr()
        return _Score(GATTN_SCORE_DOT if self.kind == "dot" else GATTN_SCORE_GATV2,
                      float(self.scale), a, float(self.neg_slope))


class Plan:
    """Per-graph plan (``gattn_plan_create``); frees its device memory on close()."""

    def __init__(self, handle, indptr_len: int):
        self._h = handle
        self._ws = {}

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan already destroyed")
        return self._h

    def info(self) -> dict:
        return gattn_plan_get_info(self)

    def workspace(self, H: int, D: int, dtype, device=None) -> torch.Tensor:
        key = (H, D, dtype)
        if key not in self._ws:
            n = gattn_workspace_size(self, H, D, dtype)
            self._ws[key] = torch.empty(max(n, 16), dtype=torch.uint8,
                                        device=device or torch.device("cuda"))
        return self._ws[key]

    def close(self):
        if self._h is not None:
            self._ws.clear()
            _check(load_library().gattn_plan_destroy(self._h), "gattn_plan_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------------------
# the C ABI, one Python function per entry point
# ----------------------------------------------------------------------------
def gattn_version() -> str:
    return load_library().gattn_version().decode()


def gattn_plan_create(indptr: torch.Tensor, indices: torch.Tensor, heavy_threshold: int = 0,
                      chunk: int = 0, stream=None, tile_enable: bool = False,
                      tile_density: float = 0.0) -> Plan:
    lib = load_library()
    for t, name in ((indptr, "indptr"), (indices, "indices")):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    opts = _PlanOpts(int(heavy_threshold), int(chunk), int(bool(tile_enable)),
                     float(tile_density))
    h = ctypes.c_void_p()
    N = indptr.numel() - 1
    _check(lib.gattn_plan_create(_ptr(indptr), _ptr(indices) if indices.numel() else None,
                                 N, indices.numel(), ctypes.byref(opts), _stream(stream),
                                 ctypes.byref(h)), "gattn_plan_create")
    return Plan(h, indptr.numel())


def gattn_plan_get_info(plan: Plan) -> dict:
    info = _PlanInfo()
    _check(load_library().gattn_plan_get_info(plan.handle, ctypes.byref(info)),
           "gattn_plan_get_info")
    return {name: getattr(info, name) for name, _ in _PlanInfo._fields_}


def gattn_plan_export(plan: Plan) -> dict:
    info = gattn_plan_get_info(plan)
    N, M = info["N"], info["M"]
    arr = {
        "deg": np.zeros(N, np.int32), "hist": np.zeros(33, np.int32),
        "light": np.zeros(info["n_light"], np.int32),
        "chunks": np.zeros((info["n_chunks"], 3), np.int32),
        "indptrT": np.zeros(N + 1, np.int32), "csc_dst": np.zeros(M, np.int32),
        "csc_eid": np.zeros(M, np.int32), "outdeg": np.zeros(N, np.int32),
        "hist_out": np.zeros(33, np.int32), "light_src": np.zeros(info["n_light_src"], np.int32),
        "src_chunks": np.zeros((info["n_src_chunks"], 3), np.int32),
    }
    order = ("deg", "hist", "light", "chunks", "indptrT", "csc_dst", "csc_eid", "outdeg",
             "hist_out", "light_src", "src_chunks")
    ptrs = [arr[k].ctypes.data_as(ctypes.c_void_p) if arr[k].size else None for k in order]
    _check(load_library().gattn_plan_export(plan.handle, *ptrs), "gattn_plan_export")
    return arr


def gattn_plan_export_tiles(plan: Plan) -> dict:
    """Dense-tile split of a plan built with tile_enable: tiles, masks, residual CSR."""
    info = gattn_plan_get_info(plan)
    nt, N = info["n_tiles"], info["N"]
    arr = {
        "tile_rb": np.zeros(nt, np.int32), "tile_cb": np.zeros(nt, np.int32),
        "masks": np.zeros((nt, 128, 4), np.uint32), "indptr_r": np.zeros(N + 1, np.int32),
        "indices_r": np.zeros(info["M"] - info["tile_edges"], np.int32),
    }
    order = ("tile_rb", "tile_cb", "masks", "indptr_r", "indices_r")
    ptrs = [arr[k].ctypes.data_as(ctypes.c_void_p) if arr[k].size else None for k in order]
    _check(load_library().gattn_plan_export_tiles(plan.handle, *ptrs), "gattn_plan_export_tiles")
    return arr


def gattn_plan_export_tile_bwd(plan: Plan) -> dict:
    """Structures of the tile backward: tiles by column block, transposed
    masks, and the residual CSC."""
    info = gattn_plan_get_info(plan)
    nt, N = info["n_tiles"], info["N"]
    lib = load_library()
    n = ctypes.c_int64(0)
    _check(lib.gattn_plan_export_tile_bwd(plan.handle, ctypes.byref(n), *([None] * 6)),
           "gattn_plan_export_tile_bwd")
    nc = int(n.value)
    arr = {
        "tcol_cb": np.zeros(nc, np.int32), "tcol_ptr": np.zeros(nc + 1, np.int32),
        "tcol_tile": np.zeros(nt, np.int32), "masks_t": np.zeros((nt, 128, 4), np.uint32),
        "indptrT_r": np.zeros(N + 1, np.int32),
        "csc_dst_r": np.zeros(info["M"] - info["tile_edges"], np.int32),
    }
    order = ("tcol_cb", "tcol_ptr", "tcol_tile", "masks_t", "indptrT_r", "csc_dst_r")
    ptrs = [arr[k].ctypes.data_as(ctypes.c_void_p) if arr[k].size else None for k in order]
    _check(lib.gattn_plan_export_tile_bwd(plan.handle, None, *ptrs), "gattn_plan_export_tile_bwd")
    return arr


REORDER = {"degree": 0, "rcm": 1}


def gattn_reorder(indptr: np.ndarray, indices: np.ndarray, kind: str = "rcm") -> np.ndarray:
    """Relabelling of a host CSR graph: perm[new] = old (host call)."""
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N = len(indptr) - 1
    perm = np.zeros(max(N, 1), np.int32)
    _check(load_library().gattn_reorder(indptr.ctypes.data, indices.ctypes.data if indices.size
                                        else None, N, int(indptr[-1]), REORDER[kind],
                                        perm.ctypes.data), "gattn_reorder")
    return perm[:N]


def gattn_permute_csr(indptr: np.ndarray, indices: np.ndarray, perm: np.ndarray):
    """The host CSR graph under a relabelling: (indptr, indices) with sorted rows."""
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    perm = np.ascontiguousarray(perm, dtype=np.int32)
    N, M = len(indptr) - 1, int(indptr[-1])
    ptr = np.zeros(N + 1, np.int32)
    idx = np.zeros(max(M, 1), np.int32)
    _check(load_library().gattn_permute_csr(indptr.ctypes.data, indices.ctypes.data if M else None,
                                            N, M, perm.ctypes.data if N else None, ptr.ctypes.data,
                                            idx.ctypes.data), "gattn_permute_csr")
    return ptr, idx[:M]


def gattn_permute_rows(x: torch.Tensor, perm: torch.Tensor, inverse: bool = False, out=None,
                       stream=None) -> torch.Tensor:
    """Rows of a CUDA tensor under perm: out[i] = x[perm[i]] (or out[perm[i]] = x[i])."""
    if not x.is_cuda or not x.is_contiguous() or perm.dtype != torch.int32 or not perm.is_cuda:
        raise ValueError("x must be a contiguous CUDA tensor and perm a CUDA int32 tensor")
    out = torch.empty_like(x) if out is None else out
    N = x.shape[0]
    row_bytes = x[0].numel() * x.element_size() if N else 16
    _check(load_library().gattn_permute_rows(_ptr(x), _ptr(out), _ptr(perm), N, row_bytes,
                                             int(bool(inverse)), _stream(stream)),
           "gattn_permute_rows")
    return out


POOL = {"max": 0, "min": 1}


def gattn_pool_workspace_size(plan: Plan, F: int, dtype) -> int:
    n = ctypes.c_size_t()
    _check(load_library().gattn_pool_workspace_size(plan.handle, F, _dtype_code(dtype),
                                                     ctypes.byref(n)), "gattn_pool_workspace_size")
    return n.value


def _pool_ws(plan: Plan, F: int, dtype, device, workspace):
    if workspace is not None:
        return workspace
    return torch.empty(gattn_pool_workspace_size(plan, F, dtype), dtype=torch.uint8,
                       device=device)


def gattn_pool_fwd(plan: Plan, x: torch.Tensor, op: str = "max", out=None, arg=None,
                   workspace=None, stream=None):
    """Max / min pooling of source rows: returns (out [N, F] in x's dtype, arg int32 [N, F])."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [N, F]")
    x2 = x.reshape(x.shape[0], -1)
    F = x2.shape[1]
    out = torch.empty_like(x2) if out is None else out
    arg = torch.empty(x2.shape, dtype=torch.int32, device=x.device) if arg is None else arg
    ws = _pool_ws(plan, F, x.dtype, x.device, workspace)
    _check(load_library().gattn_pool_fwd(plan.handle, F, _dtype_code(x.dtype), POOL[op], _ptr(x2),
                                         _ptr(out), _ptr(arg), _ptr(ws), ws.numel(),
                                         _stream(stream)), "gattn_pool_fwd")
    return out.view(x.shape), arg.view(x.shape)


def gattn_pool_bwd(plan: Plan, arg: torch.Tensor, dout: torch.Tensor, dx=None, workspace=None,
                   stream=None):
    """Gradient of pooling: dx[j] collects dout[i] wherever arg[i] == j."""
    d2 = dout.contiguous().reshape(dout.shape[0], -1)
    F = d2.shape[1]
    dx = torch.empty_like(d2) if dx is None else dx
    ws = _pool_ws(plan, F, dout.dtype, dout.device, workspace)
    _check(load_library().gattn_pool_bwd(plan.handle, F, _dtype_code(dout.dtype),
                                         _ptr(arg.contiguous()), _ptr(d2), _ptr(dx), _ptr(ws),
                                         ws.numel(), _stream(stream)), "gattn_pool_bwd")
    return dx.view(dout.shape)


def gattn_spmm_workspace_size(plan: Plan, F: int, dtype) -> int:
    n = ctypes.c_size_t()
    _check(load_library().gattn_spmm_workspace_size(plan.handle, F, _dtype_code(dtype),
                                                     ctypes.byref(n)), "gattn_spmm_workspace_size")
    return n.value


def gattn_spmm(plan: Plan, w: torch.Tensor, x: torch.Tensor, transpose: bool = False, y=None,
               workspace=None, stream=None) -> torch.Tensor:
    """y = A x (or A^T x) with edge weights w (fp32 [M], the plan's CSR order)."""
    if not x.is_cuda or not x.is_contiguous() or w.dtype != torch.float32 or not w.is_cuda:
        raise ValueError("x must be a contiguous CUDA tensor and w a CUDA fp32 tensor")
    x2 = x.reshape(x.shape[0], -1)
    F = x2.shape[1]
    y = torch.empty_like(x2) if y is None else y
    ws = workspace
    if ws is None:
        ws = torch.empty(gattn_spmm_workspace_size(plan, F, x.dtype), dtype=torch.uint8,
                         device=x.device)
    _check(load_library().gattn_spmm(plan.handle, F, _dtype_code(x.dtype), _ptr(w.contiguous()),
                                     _ptr(x2), _ptr(y), int(bool(transpose)), _ptr(ws), ws.numel(),
                                     _stream(stream)), "gattn_spmm")
    return y.view(x.shape)


def gattn_workspace_size(plan: Plan, H: int, D: int, dtype) -> int:
    n = ctypes.c_size_t()
    _check(load_library().gattn_workspace_size(plan.handle, H, D, _dtype_code(dtype),
                                                ctypes.byref(n)), "gattn_workspace_size")
    return n.value


def _shape(Q):
    if Q.dim() != 3 or not Q.is_cuda or not Q.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors of shape [N, H, D]")
    return Q.shape[1], Q.shape[2]


def gattn_fwd(plan: Plan, Q, K, V, score: Score, out=None, lse=None, workspace=None,
              stream=None):
    """Forward: returns (out [N,H,D] in Q's dtype, lse fp32 [N,H])."""
    H, D = _shape(Q)
    for t in (K, V):
        if t.shape != Q.shape or t.dtype != Q.dtype or not t.is_contiguous():
            raise ValueError("Q, K, V must share shape, dtype and be contiguous")
    out = torch.empty_like(Q) if out is None else out
    lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=Q.device) if lse is None else lse
    ws = plan.workspace(H, D, Q.dtype, Q.device) if workspace is None else workspace
    sc = score._struct()
    _check(load_library().gattn_fwd(plan.handle, H, D, _dtype_code(Q.dtype), _ptr(Q), _ptr(K),
                                    _ptr(V), ctypes.byref(sc), _ptr(out), _ptr(lse), _ptr(ws),
                                    ws.numel(), _stream(stream)), "gattn_fwd")
    return out, lse


def gattn_bwd(plan: Plan, Q, K, V, out, dout, lse, score: Score, dQ=None, dK=None, dV=None,
              da=None, workspace=None, stream=None):
    """Backward: returns (dQ, dK, dV, da) -- da is None for the dot score."""
    H, D = _shape(Q)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(Q) if dK is None else dK
    dV = torch.empty_like(Q) if dV is None else dV
    if score.kind == "gatv2" and da is None:
        da = torch.empty((H, D), dtype=torch.float32, device=Q.device)
    ws = plan.workspace(H, D, Q.dtype, Q.device) if workspace is None else workspace
    sc = score._struct()
    _check(load_library().gattn_bwd(plan.handle, H, D, _dtype_code(Q.dtype), _ptr(Q), _ptr(K),
                                    _ptr(V), ctypes.byref(sc), _ptr(out), _ptr(dout), _ptr(lse),
                                    _ptr(dQ), _ptr(dK), _ptr(dV),
                                    _ptr(da) if score.kind == "gatv2" else None, _ptr(ws),
                                    ws.numel(), _stream(stream)), "gattn_bwd")
    return dQ, dK, dV, (da if score.kind == "gatv2" else None)


def gattn_bwd_dq(plan: Plan, Q, K, V, out, dout, lse, score: Score, dQ=None, da=None,
                 workspace=None, stream=None):
    """CSR pass of the backward: returns (dQ, da); leaves Delta in the workspace."""
    H, D = _shape(Q)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    if score.kind == "gatv2" and da is None:
        da = torch.empty((H, D), dtype=torch.float32, device=Q.device)
    ws = plan.workspace(H, D, Q.dtype, Q.device) if workspace is None else workspace
    sc = score._struct()
    _check(load_library().gattn_bwd_dq(plan.handle, H, D, _dtype_code(Q.dtype), _ptr(Q), _ptr(K),
                                       _ptr(V), ctypes.byref(sc), _ptr(out), _ptr(dout),
                                       _ptr(lse), _ptr(dQ),
                                       _ptr(da) if score.kind == "gatv2" else None, _ptr(ws),
                                       ws.numel(), _stream(stream)), "gattn_bwd_dq")
    return dQ, (da if score.kind == "gatv2" else None)


def gattn_bwd_dkdv(plan: Plan, Q, K, V, dout, lse, score: Score, dK=None, dV=None,
                   workspace=None, stream=None):
    """CSC pass of the backward (after gattn_bwd_dq on the same workspace): (dK, dV)."""
    H, D = _shape(Q)
    dK = torch.empty_like(Q) if dK is None else dK
    dV = torch.empty_like(Q) if dV is None else dV
    ws = plan.workspace(H, D, Q.dtype, Q.device) if workspace is None else workspace
    sc = score._struct()
    _check(load_library().gattn_bwd_dkdv(plan.handle, H, D, _dtype_code(Q.dtype), _ptr(Q),
                                         _ptr(K), _ptr(V), ctypes.byref(sc), _ptr(dout),
                                         _ptr(lse), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(),
                                         _stream(stream)), "gattn_bwd_dkdv")
    return dK, dV


def gattn_plan_check_errors(plan: Plan) -> None:
    """Raise GattnError(GATTN_ERR_TIMEOUT) if a kernel gave up a bounded wait."""
    _check(load_library().gattn_plan_check_errors(plan.handle), "gattn_plan_check_errors")


def gattn_plan_set_wait_test(plan: Plan, fail_first_wait: bool) -> None:
    """Test hook of the bounded-wait failure path: while set, every warp of the
    attention passes run with ``plan`` gives up its first wait at once (and
    still waits for the copies it issued), so the next
    gattn_plan_check_errors raises GATTN_ERR_TIMEOUT."""
    _check(load_library().gattn_plan_set_wait_test(plan.handle, int(bool(fail_first_wait))),
           "gattn_plan_set_wait_test")


def gattn_fwd_noalloc(plan: Plan, Q, K, V, score: Score, out, lse, stream=None):
    """Forward pass that allocates nothing: ``out`` and ``lse`` must be given,
    and the heavy-chunk scratch comes from the library's fixed 32 MiB array
    (for callers that cannot allocate device memory where they run the layer,
    e.g. under an allocator or memory pool they do not own)."""
    H, D = _shape(Q)
    sc = score._struct()
    _check(load_library().gattn_fwd_noalloc(plan.handle, H, D, _dtype_code(Q.dtype), _ptr(Q),
                                            _ptr(K), _ptr(V), ctypes.byref(sc), _ptr(out),
                                            _ptr(lse), _stream(stream)), "gattn_fwd_noalloc")
    return out, lse
