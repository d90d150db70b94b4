"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every output; the five
workloads are compared in the launch configuration the benchmark uses
(default plan options): in full where the oracle finishes in seconds, else
on sampled destinations (out, lse, dQ; the largest-degree hubs included)
and sampled sources (dK, dV; the largest out-degrees included).
"""
import os

import numpy as np
import pytest

from tests import helpers as hp
from gnn_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

# (dtype, H, D): every supported row size from 32 B to 2 KB, heads of 1..32 lanes
SHAPES = [
    ("f32", 2, 4), ("f32", 2, 16), ("f32", 4, 16), ("f32", 8, 16), ("f32", 4, 64),
    ("f32", 8, 64), ("f32", 1, 128),
    ("bf16", 1, 16), ("bf16", 2, 16), ("bf16", 16, 8), ("bf16", 8, 16), ("bf16", 4, 32),
    ("bf16", 8, 64), ("bf16", 4, 128), ("bf16", 8, 128), ("bf16", 2, 256),
]


@pytest.mark.parametrize("kind", ["dot", "gatv2"])
@pytest.mark.parametrize("dtype,H,D", SHAPES)
def test_small_heavy_split(dtype, H, D, kind):
    """Hub destination and hub source, threshold/chunk 16: many chunks on
    both sides, ragged last chunks, isolated nodes."""
    indptr, indices = hp.graph_with_source_hub(5, 400, 10.0, isolated=0.05, hub_deg=333)
    case = hp.GpuCase(indptr, indices, H, D, dtype, kind, seed=11, T=16, C=16)
    try:
        got = case.run()
        hp.compare(got, hp.full_oracle(case), hp.TOL[dtype])
    finally:
        case.close()


@pytest.mark.parametrize("kind", ["dot", "gatv2"])
@pytest.mark.parametrize("dtype,H,D", SHAPES)
def test_long_items_every_row_size(dtype, H, D, kind):
    """Work items of ~40-64 edges (threshold/chunk 64): every pass takes its
    long-item stages, with the starting items' rows inline where a stage holds
    whole 4-row sets, for every row size; a hub destination and a hub source
    add chunks and merge trees."""
    indptr, indices = hp.graph_with_source_hub(7, 600, 40.0, isolated=0.03, hub_deg=500,
                                               frac=0.5)
    case = hp.GpuCase(indptr, indices, H, D, dtype, kind, seed=13, T=64, C=64)
    try:
        e = np.diff(indptr)
        assert e.sum() / max(1, len(e)) > 16           # mean item above the short-item bar
        hp.compare(case.run(), hp.full_oracle(case), hp.TOL[dtype])
    finally:
        case.close()


@pytest.mark.parametrize("kind", ["dot", "gatv2"])
@pytest.mark.parametrize("dtype,H,D", [("f32", 2, 16), ("bf16", 8, 16), ("bf16", 4, 32),
                                       ("bf16", 8, 64)])
def test_default_plan(dtype, H, D, kind):
    indptr, indices = hp.graph_with_source_hub(6, 2000, 30.0, isolated=0.02, hub_deg=1500,
                                               frac=0.3)
    case = hp.GpuCase(indptr, indices, H, D, dtype, kind, seed=12)
    try:
        hp.compare(case.run(), hp.full_oracle(case), hp.TOL[dtype])
    finally:
        case.close()


@pytest.mark.parametrize("deg", [1, 15, 16, 17, 31, 32, 33, 47, 64, 65])
def test_ragged_degrees(deg):
    """Every row has the same degree around the 16-edge chunk and 32-edge
    index-batch boundaries."""
    N = 120
    r = np.random.default_rng(deg)
    rows = [np.sort(r.choice(np.setdiff1d(np.arange(N), [i]), deg, replace=False))
            for i in range(N)]
    indptr = np.arange(N + 1, dtype=np.int32) * deg
    indices = np.concatenate(rows).astype(np.int32)
    for T, C in ((0, 0), (16, 16)):
        case = hp.GpuCase(indptr, indices, 4, 32, "bf16", "dot", seed=deg, T=T, C=C)
        try:
            hp.compare(case.run(), hp.full_oracle(case), hp.TOL["bf16"])
        finally:
            case.close()


def test_edge_cases():
    cases = []
    # all isolated
    cases.append((np.zeros(6, np.int32), np.zeros(0, np.int32)))
    # a single node with a self-loop
    cases.append((np.array([0, 1], np.int32), np.array([0], np.int32)))
    # multi-edges and unsorted rows
    cases.append((np.array([0, 4, 4, 7], np.int32), np.array([2, 1, 2, 2, 0, 0, 1], np.int32)))
    # one star: node 0 receives from everyone, everyone else isolated
    n = 3000
    cases.append((np.concatenate([[0], np.full(n, n - 1)]).astype(np.int32),
                  np.arange(1, n, dtype=np.int32)))
    for indptr, indices in cases:
        for kind in ("dot", "gatv2"):
            for T in (0, 2):
                case = hp.GpuCase(indptr, indices, 2, 16, "f32", kind, seed=3, T=T, C=T)
                try:
                    hp.compare(case.run(), hp.full_oracle(case), hp.TOL["f32"])
                finally:
                    case.close()


def test_deterministic_and_allocation_free():
    indptr, indices = hp.graph_with_source_hub(7, 3000, 20.0, hub_deg=2500)
    case = hp.GpuCase(indptr, indices, 4, 32, "bf16", "gatv2", seed=5, T=64, C=64)
    try:
        first = case.run()
        free0 = torch.cuda.mem_get_info()[0]
        alloc0 = torch.cuda.memory_allocated()
        # reuse outputs: nothing may be allocated by the library
        from gnn_sparse_attention_gb300 import binding as gb
        Q, K, V, G = (case.t[k] for k in ("Q", "K", "V", "dO"))
        out = torch.empty_like(Q)
        lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=Q.device)
        dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))
        da = torch.empty_like(case.a)
        alloc1 = torch.cuda.memory_allocated()
        free1 = torch.cuda.mem_get_info()[0]
        gb.gattn_fwd(case.plan, Q, K, V, case.score, out=out, lse=lse)
        gb.gattn_bwd(case.plan, Q, K, V, out, G, lse, case.score, dQ=dQ, dK=dK, dV=dV, da=da)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free1
        assert torch.cuda.memory_allocated() == alloc1
        for k, t in (("out", out), ("lse", lse), ("dQ", dQ), ("dK", dK), ("dV", dV), ("da", da)):
            assert torch.equal(t, first[k]), f"{k} not bitwise reproducible"
        del free0, alloc0
    finally:
        case.close()


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
def _workload_case(name):
    w = synth.WORKLOADS[name]
    indptr, indices = hp.workload_graph(name)
    return hp.GpuCase(indptr, indices, w.H, w.D, w.dtype, w.score, seed=0)


def test_er1k_full():
    case = _workload_case("er1k")
    try:
        hp.compare(case.run(), hp.full_oracle(case), hp.TOL["f32"])
    finally:
        case.close()


def test_powerlaw170k_full():
    case = _workload_case("powerlaw170k")
    try:
        hp.compare(case.run(), hp.full_oracle(case), hp.TOL["bf16"])
    finally:
        case.close()


def _sample(indptr, indices, seed, n_rows=160, n_src=12):
    r = np.random.default_rng(seed)
    N = len(indptr) - 1
    deg = np.diff(indptr)
    outdeg = np.bincount(indices, minlength=N)
    top = np.argsort(-deg, kind="stable")[:8]
    rows = np.unique(np.concatenate([top, r.choice(N, n_rows, replace=False),
                                     np.nonzero(deg == 0)[0][:4]]))
    has_out = np.nonzero(outdeg > 0)[0]
    srcs = np.unique(np.concatenate([np.argsort(-outdeg, kind="stable")[:3],
                                     r.choice(has_out, n_src, replace=False)]))
    zero_src = np.nonzero(outdeg == 0)[0][:4]
    return rows, srcs, zero_src


@pytest.mark.parametrize("name", ["lognormal233k", "gatv2_powerlaw2m4", "sbm1m"])
def test_large_workload_sampled(name):
    case = _workload_case(name)
    try:
        got = case.run()
        rows, srcs, zero_src = _sample(case.indptr, case.indices, 1)
        if name != "sbm1m":
            # at least 200 sources for dK/dV: those with the cheapest oracle
            # closure among 2000 random ones, the largest out-degrees, and
            # (where the plan has both kinds) light and heavy sources alike
            srcs = np.union1d(srcs, hp.cheap_sources(case.indptr, case.indices, 2))
            T = case.plan.info()["heavy_threshold"]
            outdeg = np.bincount(case.indices, minlength=len(case.indptr) - 1)
            heavy = outdeg[srcs] > T
            assert len(srcs) >= 200
            assert heavy.any() or not (outdeg > T).any()
            assert (~heavy).any() or not ((outdeg > 0) & (outdeg <= T)).any()
        ref = hp.sampled_oracle(case, rows, srcs, group=8, threads=min(8, os.cpu_count() or 1))
        tol = hp.TOL[case.dtype]
        e1 = hp.compare({k: got[k] for k in ("out", "lse", "dQ")}, ref["rows"], tol, rows=rows)
        e2 = hp.compare({k: got[k] for k in ("dK", "dV")}, ref["srcs"], tol, rows=srcs)
        for k in ("dK", "dV"):
            assert np.all(hp.to64(got[k], zero_src) == 0)
        # properties over every output: finite everywhere, lse = -inf exactly
        # on isolated nodes, and out = 0 there
        deg = np.diff(case.indptr)
        lse = got["lse"].cpu().numpy()
        assert np.array_equal(np.isneginf(lse).any(axis=1), deg == 0)
        for k in ("out", "dQ", "dK", "dV"):
            assert torch.isfinite(got[k].float()).all(), k
        print(name, e1, e2)
    finally:
        case.close()


def test_gatv2_powerlaw2m4_da_full():
    """da is one sum over all 62M edges: checked against the full oracle."""
    import oracle
    case = _workload_case("gatv2_powerlaw2m4")
    try:
        got = case.run()
        Q, K, V, G = (case.host64(k) for k in ("Q", "K", "V", "dO"))
        _, _, _, da = oracle.backward(case.indptr, case.indices, Q, K, V, G, kind=oracle.GATV2,
                                      a=case.a64)
        err = hp.relerr(hp.to64(got["da"]), da)
        assert err <= hp.TOL["bf16"], err
    finally:
        case.close()
