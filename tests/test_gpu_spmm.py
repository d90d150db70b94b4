"""Weighted SpMM on the GPU through the C ABI against the oracle: the CSR
pass (light rows, heavy rows over merge trees), the transposed product over
the cached CSC, and the weighted block-sparse tensor-core path of tiled
plans."""
import numpy as np
import pytest

import oracle
from gnn_sparse_attention_gb300 import synth
from tests.helpers import TOL, relerr

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

pytestmark = pytest.mark.gpu

from gnn_sparse_attention_gb300 import binding as gb  # noqa: E402


def _sbm(N, seed):
    w = synth.Workload("sbm_case", "sbm", N, 1, 64, "bf16", "dot", False,
                       {"block": 64, "p_in": 0.5, "inter_per_node": 4})
    return synth.make_graph(w, seed=seed)


def _run(ip, ix, W, X, dtype, transpose=False, T=0, C=0, tile=False):
    dev = torch.device("cuda")
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    plan = gb.gattn_plan_create(torch.from_numpy(ip).to(dev), torch.from_numpy(ix).to(dev), T, C,
                                tile_enable=tile)
    try:
        x = torch.from_numpy(np.ascontiguousarray(X, np.float32)).to(dev, tdt)
        w = torch.from_numpy(np.ascontiguousarray(W, np.float32)).to(dev)
        y = gb.gattn_spmm(plan, w, x, transpose=transpose)
        torch.cuda.synchronize()
        gb.gattn_plan_check_errors(plan)
        return y.double().cpu().numpy(), x.double().cpu().numpy(), plan.info()
    finally:
        plan.close()


def _graph(seed, N=800):
    ip, ix = synth.small_graph(seed, N, 8.0, isolated=0.05, hub_deg=600)
    rows = [list(ix[ip[i]:ip[i + 1]]) for i in range(N)]
    rows[3] += rows[3][:5]                                     # repeated edges
    ip = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    return ip, np.array([j for r in rows for j in r], np.int32)


@pytest.mark.parametrize("dtype,F", [("f32", 8), ("f32", 128), ("bf16", 16), ("bf16", 256),
                                     ("bf16", 1024)])
@pytest.mark.parametrize("transpose", [False, True])
def test_spmm_csr_matches_oracle(dtype, F, transpose):
    ip, ix = _graph(31 + F)
    r = np.random.default_rng(F)
    W = r.standard_normal(len(ix))
    X = r.standard_normal((len(ip) - 1, F))
    y, x64, _ = _run(ip, ix, W, X, dtype, transpose=transpose, T=16, C=16)
    w64 = W.astype(np.float32).astype(np.float64)
    if transpose:
        pl = oracle.plan(ip, ix, 16, 16)
        ref = oracle.spmm(pl["indptrT"], pl["csc_dst"], w64[pl["csc_eid"]], x64)
    else:
        ref = oracle.spmm(ip, ix, w64, x64)
    assert relerr(y, ref) <= TOL[dtype]


@pytest.mark.parametrize("N,F", [(1000, 64), (777, 128), (1024, 256), (640, 512)])
def test_spmm_wsb_tiles_match_oracle(N, F):
    ip, ix = _sbm(N, seed=N)
    r = np.random.default_rng(N)
    W = r.uniform(0.1, 1.0, len(ix))
    X = r.standard_normal((N, F))
    y, x64, info = _run(ip, ix, W, X, "bf16", tile=True)
    assert info["n_tiles"] > 0 and info["tile_edges"] > 0
    ref = oracle.spmm(ip, ix, W.astype(np.float32).astype(np.float64), x64)
    assert relerr(y, ref) <= TOL["bf16"]
    y2, _, _ = _run(ip, ix, W, X, "bf16")              # the same product on the CSR pass
    assert relerr(y, y2) <= TOL["bf16"]


@pytest.mark.slow
def test_spmm_sbm1m_wsb_sampled():
    w = synth.WORKLOADS["sbm1m"]
    ip, ix = synth.make_graph(w, seed=0)
    r = np.random.default_rng(0)
    W = r.uniform(0.1, 1.0, len(ix))
    X = synth.normal(0, 1, (w.N, 128))
    y, x64, info = _run(ip, ix, W, X, "bf16", tile=True)
    assert info["n_tile_rows"] == w.N // 128
    rows = np.unique(np.concatenate([r.integers(0, w.N, 300), [0, 127, 128, w.N - 1]]))
    rp, col, _ = oracle.rows_subgraph(ip, ix, rows)
    eid = np.concatenate([np.arange(ip[i], ip[i + 1]) for i in rows])
    ref = oracle.spmm(rp, col, W.astype(np.float32).astype(np.float64)[eid], x64)
    assert relerr(y[rows], ref) <= TOL["bf16"]
