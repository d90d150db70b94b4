"""fp64 CPU oracle for fused CSR graph attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

The arithmetic lives in ``gattn_oracle.c`` (plain loops, fp64, serial); this
module only compiles it with gcc, marshals numpy arrays through ctypes and
offers a row-subset helper so that single outputs of a large graph can be
computed one by one.

What is computed, and where it comes from ("On Efficient Scaling of GNNs via
IO-Aware Layers Implementations", zh/ko technical summaries, "Methodology",
attention-based layers): per destination node a softmax over its
in-neighbours' scores, the weighted sum of their values and a per-node
log-sum-exp; the backward is the analytic gradient of that softmax attention.
Every function is pinned by the CPU tests in ``tests/test_oracle_pins.py``
(dense brute force, closed forms, finite differences, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gattn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DOT = 0
GATV2 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: fp64 as written)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.oracle_forward.argtypes = [i64, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           dbl, P, dbl, P, P, P, P, P]
            lib.oracle_forward.restype = ctypes.c_int
            lib.oracle_backward.argtypes = [i64, P, P, P, i64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, dbl, P, dbl, P, P, P, P, P, P, P, P]
            lib.oracle_backward.restype = ctypes.c_int
            lib.oracle_plan.argtypes = [i32, i64, P, P, i32, i32, P, P, P, P, i64, P, P, P, P, P,
                                        P, P, i64, P]
            lib.oracle_plan.restype = ctypes.c_int
            lib.oracle_tile_plan.argtypes = [i32, i64, P, P, i64, i64, P, P, P, P, P, P]
            lib.oracle_tile_plan.restype = ctypes.c_int
            lib.oracle_spmm.argtypes = [i64, P, P, P, i64, P, P]
            lib.oracle_spmm.restype = ctypes.c_int
            lib.oracle_reduce_forward.argtypes = [i64, P, P, i64, ctypes.c_int, P, P, P]
            lib.oracle_reduce_forward.restype = ctypes.c_int
            lib.oracle_reduce_backward.argtypes = [i64, i64, i64, P, P, P]
            lib.oracle_reduce_backward.restype = ctypes.c_int
            lib.oracle_reorder.argtypes = [i32, i64, P, P, ctypes.c_int, P]
            lib.oracle_reorder.restype = ctypes.c_int
            lib.oracle_permute_csr.argtypes = [i32, i64, P, P, P, P, P]
            lib.oracle_permute_csr.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _rows_args(indptr, indices, rows):
    row_ptr = np.ascontiguousarray(indptr, dtype=np.int64)
    col = np.ascontiguousarray(indices, dtype=np.int32)
    row_ids = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n_rows = len(row_ptr) - 1
    return n_rows, row_ids, row_ptr, col


def _score_args(kind, D, scale, a):
    if kind == DOT:
        return (1.0 / np.sqrt(D) if scale is None else float(scale)), None
    if a is None:
        raise ValueError("GATv2 needs the attention vector a[H, D]")
    return 0.0, _f64(a)


def forward(indptr, indices, Q, K, V, kind=DOT, scale=None, a=None, slope=0.2, rows=None):
    """Oracle forward.  Q, K, V: [N, H, D] (any float dtype, converted to fp64).

    ``indptr``/``indices`` describe destination rows; with ``rows`` given,
    row r is node ``rows[r]`` (a subset of the graph's rows, each complete).
    Returns (out [n_rows, H, D], lse [n_rows, H]) in fp64.
    """
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    _, H, D = Q.shape
    n_rows, row_ids, row_ptr, col = _rows_args(indptr, indices, rows)
    sc, a64 = _score_args(kind, D, scale, a)
    out = np.zeros((n_rows, H, D), np.float64)
    lse = np.zeros((n_rows, H), np.float64)
    rc = lib.oracle_forward(n_rows, _p(row_ids), _p(row_ptr), _p(col), H, D, kind, sc, _p(a64),
                            float(slope), _p(Q), _p(K), _p(V), _p(out), _p(lse))
    if rc != 0:
        raise MemoryError("oracle_forward failed")
    return out, lse


def backward(indptr, indices, Q, K, V, dO, kind=DOT, scale=None, a=None, slope=0.2, rows=None):
    """Oracle analytic backward of L = sum(out * dO).

    dO is given per row position.  Returns (dQ [n_rows,H,D], dK [N,H,D],
    dV [N,H,D], da [H,D] or None).  With a row subset, dK/dV hold only the
    contributions of the listed rows' edges.
    """
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    N, H, D = K.shape
    n_rows, row_ids, row_ptr, col = _rows_args(indptr, indices, rows)
    sc, a64 = _score_args(kind, D, scale, a)
    dQ = np.zeros((n_rows, H, D), np.float64)
    dK = np.zeros((N, H, D), np.float64)
    dV = np.zeros((N, H, D), np.float64)
    da = np.zeros((H, D), np.float64) if kind == GATV2 else None
    rc = lib.oracle_backward(n_rows, _p(row_ids), _p(row_ptr), _p(col), N, H, D, kind, sc,
                             _p(a64), float(slope), _p(Q), _p(K), _p(V), _p(dO), _p(dQ), _p(dK),
                             _p(dV), _p(da))
    if rc != 0:
        raise MemoryError("oracle_backward failed")
    return dQ, dK, dV, da


def plan(indptr, indices, heavy_threshold, chunk):
    """Oracle plan (integer metadata of the light/heavy partition and CSC)."""
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N = len(indptr) - 1
    M = int(indptr[-1])
    T, C = int(heavy_threshold), int(chunk)
    cap = M // C + N + 1
    deg = np.zeros(N, np.int32)
    hist = np.zeros(33, np.int32)
    light = np.zeros(max(N, 1), np.int32)
    chunks = np.zeros((cap, 3), np.int32)
    indptrT = np.zeros(N + 1, np.int32)
    csc_dst = np.zeros(max(M, 1), np.int32)
    csc_eid = np.zeros(max(M, 1), np.int32)
    outdeg = np.zeros(N, np.int32)
    hist_out = np.zeros(33, np.int32)
    light_src = np.zeros(max(N, 1), np.int32)
    src_chunks = np.zeros((cap, 3), np.int32)
    counts = np.zeros(4, np.int64)
    rc = lib.oracle_plan(N, M, _p(indptr), _p(indices), T, C, _p(deg), _p(hist), _p(light),
                         _p(chunks), cap, _p(indptrT), _p(csc_dst), _p(csc_eid), _p(outdeg),
                         _p(hist_out), _p(light_src), _p(src_chunks), cap, _p(counts))
    if rc != 0:
        raise RuntimeError(f"oracle_plan failed ({rc})")
    nl, nc, nls, ncs = (int(c) for c in counts)
    return {
        "deg": deg, "hist": hist, "light": light[:nl], "chunks": chunks[:nc],
        "indptrT": indptrT, "csc_dst": csc_dst[:M], "csc_eid": csc_eid[:M],
        "outdeg": outdeg, "hist_out": hist_out, "light_src": light_src[:nls],
        "src_chunks": src_chunks[:ncs],
    }


def spmm(indptr, indices, w, X):
    """y = A x with A the weighted adjacency (w[e] per CSR edge): [N, F] fp64."""
    lib = _load()
    X = _f64(X)
    F = int(np.prod(X.shape[1:])) if X.ndim > 1 else 1
    row_ptr = np.ascontiguousarray(indptr, dtype=np.int64)
    col = np.ascontiguousarray(indices, dtype=np.int32)
    w = _f64(w)
    n_rows = len(row_ptr) - 1
    y = np.zeros((n_rows, F), np.float64)
    lib.oracle_spmm(n_rows, _p(row_ptr), _p(col), _p(w), F, _p(X), _p(y))
    return y


MAX = 0
MIN = 1


def reduce_forward(indptr, indices, X, op=MAX, rows=None):
    """Max / min pooling of source rows over each row's edges: (out [R, F] fp64, arg [R, F] int32).

    X is [N, ...] (flattened to F features per node); ``rows`` as for forward().
    """
    lib = _load()
    X = _f64(X)
    N = X.shape[0]
    F = int(np.prod(X.shape[1:])) if X.ndim > 1 else 1
    n_rows, row_ids, row_ptr, col = _rows_args(indptr, indices, rows)
    out = np.zeros((n_rows, F), np.float64)
    arg = np.zeros((n_rows, F), np.int32)
    rc = lib.oracle_reduce_forward(n_rows, _p(row_ptr), _p(col), F, int(op), _p(X), _p(out),
                                   _p(arg))
    if rc != 0:
        raise RuntimeError(f"oracle_reduce_forward failed ({rc})")
    return out, arg


def reduce_backward(arg, dout, N):
    """dx [N, F] of max / min pooling: each row's gradient goes to its arg source."""
    lib = _load()
    arg = np.ascontiguousarray(arg, dtype=np.int32)
    dout = _f64(dout).reshape(arg.shape)
    F = arg.shape[1]
    dx = np.zeros((N, F), np.float64)
    lib.oracle_reduce_backward(arg.shape[0], N, F, _p(arg), _p(dout), _p(dx))
    return dx


REORDER_DEGREE = 0
REORDER_RCM = 1


def reorder(indptr, indices, method):
    """Oracle relabelling: perm[new] = old (degree order or reverse Cuthill-McKee)."""
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N = len(indptr) - 1
    perm = np.zeros(max(N, 1), np.int32)
    rc = lib.oracle_reorder(N, int(indptr[-1]), _p(indptr), _p(indices), int(method), _p(perm))
    if rc != 0:
        raise RuntimeError(f"oracle_reorder failed ({rc})")
    return perm[:N]


def permute_csr(indptr, indices, perm):
    """Oracle relabelled graph: row i = old row perm[i], sources renamed and sorted."""
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    perm = np.ascontiguousarray(perm, dtype=np.int32)
    N = len(indptr) - 1
    M = int(indptr[-1])
    ptr = np.zeros(N + 1, np.int32)
    idx = np.zeros(max(M, 1), np.int32)
    rc = lib.oracle_permute_csr(N, M, _p(indptr), _p(indices), _p(perm), _p(ptr), _p(idx))
    if rc != 0:
        raise RuntimeError(f"oracle_permute_csr failed ({rc})")
    return ptr, idx[:M]


TILE = 128  # nodes per tile side


def tile_min_count(density: float) -> int:
    """Edges a 128 x 128 block needs to be a dense tile: ceil(density * 128^2), at least 1."""
    import math
    return max(1, int(math.ceil(float(np.float32(density)) * TILE * TILE)))


def tile_plan(indptr, indices, min_count):
    """Oracle dense-tile split: tiles (rb, cb), their bit masks and the residual CSR."""
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N = len(indptr) - 1
    M = int(indptr[-1])
    cap = M // max(int(min_count), 1) + 1
    tile_rb = np.zeros(cap, np.int32)
    tile_cb = np.zeros(cap, np.int32)
    masks = np.zeros((cap, 128, 4), np.uint32)
    indptr_r = np.zeros(N + 1, np.int32)
    indices_r = np.zeros(max(M, 1), np.int32)
    counts = np.zeros(2, np.int64)
    rc = lib.oracle_tile_plan(N, M, _p(indptr), _p(indices), int(min_count), cap, _p(tile_rb),
                              _p(tile_cb), _p(masks), _p(indptr_r), _p(indices_r), _p(counts))
    if rc != 0:
        raise RuntimeError(f"oracle_tile_plan failed ({rc})")
    nt, mr = int(counts[0]), int(counts[1])
    return {"tile_rb": tile_rb[:nt], "tile_cb": tile_cb[:nt], "masks": masks[:nt],
            "indptr_r": indptr_r, "indices_r": indices_r[:mr]}


def rows_subgraph(indptr, indices, rows):
    """CSR of a subset of destination rows (each row complete, global ids).

    Returns (row_ptr, col, rows) to pass as (indptr, indices, rows=rows).
    """
    indptr = np.asarray(indptr, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    deg = indptr[rows + 1] - indptr[rows]
    row_ptr = np.zeros(len(rows) + 1, np.int64)
    np.cumsum(deg, out=row_ptr[1:])
    if len(rows):
        starts = np.repeat(indptr[rows] - row_ptr[:-1], deg)
        col = np.asarray(indices)[np.arange(row_ptr[-1]) + starts]
    else:
        col = np.zeros(0, np.int32)
    return row_ptr, np.ascontiguousarray(col, dtype=np.int32), rows.astype(np.int32)


def sources_closure(indptr, indices, sources):
    """Destination rows that have at least one in-edge from ``sources``.

    Running the backward on those complete rows yields the exact dK/dV of
    every node in ``sources`` (all of its out-edges are covered).
    """
    mark = np.zeros(len(indptr) - 1, bool)
    mark[np.asarray(sources)] = True
    hit = mark[np.asarray(indices)]
    rows_of_edge = np.repeat(np.arange(len(indptr) - 1), np.diff(np.asarray(indptr)))
    return np.unique(rows_of_edge[hit])


class _Variant:
    """Context manager that swaps in another build of the oracle library.

    Used only by the mutation tests, which compile deliberately broken copies
    of ``gattn_oracle.c`` to show that the pins catch each planted mistake.
    """

    def __init__(self, source_text: str, tag: str):
        import tempfile
        self._dir = tempfile.mkdtemp(prefix=f"oracle_{tag}_")
        src = os.path.join(self._dir, "v.c")
        with open(src, "w") as f:
            f.write(source_text)
        self.path = os.path.join(self._dir, "v.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", src, "-o",
                               self.path, "-lm"])

    def __enter__(self):
        global _lib
        self._saved = _load()
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_forward", "oracle_backward", "oracle_plan"):
            getattr(lib, name).argtypes = getattr(self._saved, name).argtypes
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        import shutil
        shutil.rmtree(self._dir, ignore_errors=True)
        return False


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def variant(source_text: str, tag: str) -> _Variant:
    return _Variant(source_text, tag)
