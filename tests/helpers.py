"""Shared helpers of the parity tests: seeded inputs, GPU calls, oracle calls,
sampling and the error metric.

Error metric (one number per tensor): max |got - ref| / max |ref|, i.e. the
inf-norm relative error; bars 1e-4 for fp32 I/O and 2e-2 for bf16 I/O with
fp32 accumulation.
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
from gnn_sparse_attention_gb300 import synth

TOL = {"f32": 1e-4, "bf16": 2e-2}


def relerr(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    den = max(float(np.abs(ref).max()), 1e-30)
    return float(np.abs(got - ref).max()) / den


def torch_dtype(name):
    import torch
    return torch.float32 if name == "f32" else torch.bfloat16


@functools.lru_cache(maxsize=4)
def workload_graph(name: str):
    g = synth.make_graph(synth.WORKLOADS[name])
    for a in g:
        a.setflags(write=False)
    return g


def graph_with_source_hub(seed, N, avg, hub_src=1, frac=0.7, **kw):
    """small_graph plus node ``hub_src`` added as a source of ``frac`` of the rows
    (a heavy column of the transpose); rows stay sorted and duplicate-free."""
    indptr, indices = synth.small_graph(seed, N, avg, **kw)
    r = np.random.default_rng(seed + 77)
    rows = []
    for i in range(N):
        s = set(indices[indptr[i]:indptr[i + 1]].tolist())
        if i != hub_src and r.random() < frac:
            s.add(hub_src)
        rows.append(sorted(s))
    new_ptr = np.zeros(N + 1, np.int64)
    np.cumsum([len(x) for x in rows], out=new_ptr[1:])
    new_idx = np.array([j for x in rows for j in x], np.int32)
    return new_ptr.astype(np.int32), new_idx


class GpuCase:
    """Inputs on the GPU (in the I/O dtype) and their exact fp64 decodes."""

    def __init__(self, indptr, indices, H, D, dtype, kind, seed=0, T=0, C=0, feats=None,
                 tile=False, density=0.0):
        import torch
        from gnn_sparse_attention_gb300 import binding as gb
        self.indptr, self.indices = indptr, indices
        self.N = len(indptr) - 1
        self.H, self.D, self.dtype, self.kind = H, D, dtype, kind
        w = synth.Workload("case", "er", self.N, H, D, dtype, kind)
        f = feats if feats is not None else synth.make_features(w, seed=seed)
        dev = torch.device("cuda")
        tdt = torch_dtype(dtype)
        self.t = {k: torch.from_numpy(np.ascontiguousarray(f[k])).to(dev, tdt)
                  for k in ("Q", "K", "V", "dO")}
        self.a64 = f.get("a")
        self.a = torch.from_numpy(f["a"]).to(dev) if kind == "gatv2" else None
        self.score = gb.Score(kind, a=self.a)
        self.plan = gb.gattn_plan_create(torch.from_numpy(indptr).to(dev),
                                         torch.from_numpy(indices).to(dev), T, C,
                                         tile_enable=tile, tile_density=density)
        self.okind = oracle.DOT if kind == "dot" else oracle.GATV2

    def host64(self, name, rows=None):
        t = self.t[name]
        if rows is not None:
            import torch
            t = t[torch.as_tensor(rows, device=t.device, dtype=torch.long)]
        return t.double().cpu().numpy()

    def run(self):
        import torch
        from gnn_sparse_attention_gb300 import binding as gb
        Q, K, V, G = (self.t[k] for k in ("Q", "K", "V", "dO"))
        out, lse = gb.gattn_fwd(self.plan, Q, K, V, self.score)
        dQ, dK, dV, da = gb.gattn_bwd(self.plan, Q, K, V, out, G, lse, self.score)
        torch.cuda.synchronize()
        gb.gattn_plan_check_errors(self.plan)
        self.out_t = out
        return {"out": out, "lse": lse, "dQ": dQ, "dK": dK, "dV": dV, "da": da}

    def close(self):
        self.plan.close()


def to64(x, rows=None):
    import torch
    if x is None:
        return None
    if rows is not None:
        x = x[torch.as_tensor(rows, device=x.device, dtype=torch.long)]
    return x.double().cpu().numpy()


def full_oracle(case: GpuCase):
    Q, K, V, G = (case.host64(k) for k in ("Q", "K", "V", "dO"))
    out, lse = oracle.forward(case.indptr, case.indices, Q, K, V, kind=case.okind, a=case.a64)
    dQ, dK, dV, da = oracle.backward(case.indptr, case.indices, Q, K, V, G, kind=case.okind,
                                     a=case.a64)
    return {"out": out, "lse": lse, "dQ": dQ, "dK": dK, "dV": dV, "da": da}


def compare(got: dict, ref: dict, tol: float, rows=None):
    """Per-tensor inf-norm relative errors; lse compared on finite entries and
    -inf checked exactly."""
    errs = {}
    for k in ("out", "lse", "dQ", "dK", "dV", "da"):
        if ref.get(k) is None or got.get(k) is None:
            continue
        g = to64(got[k], rows) if rows is not None and k != "da" else to64(got[k])
        r = ref[k]
        if k == "lse":
            fin = np.isfinite(r)
            assert np.array_equal(np.isneginf(g), ~fin), "lse -inf pattern differs"
            g, r = g[fin], r[fin]
        errs[k] = relerr(g, r)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"parity failed (tol {tol}): {errs}"
    return errs


def compact_subgraph(indptr, indices, rows):
    """Row subset with node ids compacted to the nodes it touches.

    Returns (row_ptr, col, row_ids, nodes): row r of the subset is compact node
    row_ids[r]; compact node c is global node nodes[c].
    """
    row_ptr, col, rows = oracle.rows_subgraph(indptr, indices, rows)
    nodes, inv = np.unique(np.concatenate([rows, col]), return_inverse=True)
    row_ids = inv[:len(rows)].astype(np.int32)
    col_c = inv[len(rows):].astype(np.int32)
    return row_ptr, col_c, row_ids, nodes


def _sources_oracle(case: GpuCase, src_nodes, rows_of_edge=None):
    """Oracle dK/dV of ``src_nodes``: the backward over every destination row
    that holds one of their out-edges (all of those rows, complete)."""
    if rows_of_edge is None:
        closure = oracle.sources_closure(case.indptr, case.indices, src_nodes)
    else:  # the same rows, with the edge -> row map computed once by the caller
        mark = np.zeros(len(case.indptr) - 1, bool)
        mark[np.asarray(src_nodes)] = True
        closure = np.unique(rows_of_edge[mark[case.indices]])
    rp, col, rid, nodes = compact_subgraph(case.indptr, case.indices, closure)
    Q, K, V = (case.host64(k, nodes) for k in ("Q", "K", "V"))
    G = case.host64("dO", closure)
    _, dK, dV, _ = oracle.backward(rp, col, Q, K, V, G, kind=case.okind, a=case.a64, rows=rid)
    pos = np.searchsorted(nodes, np.asarray(src_nodes))
    return dK[pos], dV[pos]


def sampled_oracle(case: GpuCase, dst_rows, src_nodes, group=0, threads=1):
    """Oracle values of out/lse/dQ on ``dst_rows`` and dK/dV on ``src_nodes``.

    With ``group`` > 0 the sources are split into groups of that many, each
    group's closure is evaluated on its own, and ``threads`` groups run at
    once (the oracle is C called through ctypes, which releases the
    interpreter lock)."""
    res = {}
    rp, col, rid, nodes = compact_subgraph(case.indptr, case.indices, dst_rows)
    Q, K, V = (case.host64(k, nodes) for k in ("Q", "K", "V"))
    G = case.host64("dO", np.asarray(dst_rows))
    out, lse = oracle.forward(rp, col, Q, K, V, kind=case.okind, a=case.a64, rows=rid)
    dQ, _, _, _ = oracle.backward(rp, col, Q, K, V, G, kind=case.okind, a=case.a64, rows=rid)
    res["rows"] = {"out": out, "lse": lse, "dQ": dQ}
    src_nodes = np.asarray(src_nodes)
    if group <= 0:
        dK, dV = _sources_oracle(case, src_nodes)
    else:
        from concurrent.futures import ThreadPoolExecutor
        parts = [src_nodes[k:k + group] for k in range(0, len(src_nodes), group)]
        roe = np.repeat(np.arange(len(case.indptr) - 1), np.diff(np.asarray(case.indptr)))
        with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
            got = list(ex.map(lambda g: _sources_oracle(case, g, roe), parts))
        dK = np.concatenate([x[0] for x in got])
        dV = np.concatenate([x[1] for x in got])
    res["srcs"] = {"dK": dK, "dV": dV}
    return res


def cheap_sources(indptr, indices, seed, n=200, candidates=2000, top=3):
    """Sources for a sampled dK/dV check of a large graph: ``n`` of ``candidates``
    random sources (with out-edges) whose oracle closure -- the total in-degree
    of their out-neighbours -- is smallest, plus the ``top`` sources of largest
    out-degree.  Sorted, distinct."""
    r = np.random.default_rng(seed)
    N = len(indptr) - 1
    deg = np.diff(np.asarray(indptr, np.int64))
    outdeg = np.bincount(indices, minlength=N)
    cost = np.bincount(indices, weights=np.repeat(deg, deg).astype(np.float64), minlength=N)
    has_out = np.nonzero(outdeg > 0)[0]
    cand = r.choice(has_out, min(candidates, len(has_out)), replace=False)
    pick = cand[np.argsort(cost[cand], kind="stable")[:n]]
    return np.unique(np.concatenate([np.argsort(-outdeg, kind="stable")[:top], pick]))
