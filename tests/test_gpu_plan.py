"""GPU plan builder: bit-exact against the oracle's plan, and the CSR checks."""
import numpy as np
import pytest

import oracle
from tests import helpers as hp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gnn_sparse_attention_gb300 import binding as gb  # noqa: E402


def _plan_on_gpu(indptr, indices, T, C):
    dev = torch.device("cuda")
    return gb.gattn_plan_create(torch.from_numpy(np.ascontiguousarray(indptr)).to(dev),
                                torch.from_numpy(np.ascontiguousarray(indices)).to(dev), T, C)


def _assert_plan_equal(indptr, indices, T, C):
    plan = _plan_on_gpu(indptr, indices, T, C)
    try:
        info = plan.info()
        got = gb.gattn_plan_export(plan)
    finally:
        plan.close()
    ref = oracle.plan(indptr, indices, info["heavy_threshold"], info["chunk"])
    for k, v in ref.items():
        np.testing.assert_array_equal(got[k], v, err_msg=k)
    deg = np.diff(np.asarray(indptr, np.int64))
    assert info["max_deg"] == (deg.max() if len(deg) else 0)
    assert info["n_heavy"] == int((deg > info["heavy_threshold"]).sum())
    return info


@pytest.mark.parametrize("seed,N,avg,T,C", [(1, 500, 8.0, 16, 16), (2, 3000, 25.0, 64, 32),
                                            (3, 200, 2.0, 1, 1), (4, 1000, 40.0, 0, 0)])
def test_plan_small(seed, N, avg, T, C):
    indptr, indices = hp.graph_with_source_hub(seed, N, avg, isolated=0.05, hub_deg=N - 1)
    r = np.random.default_rng(seed)
    indices = indices.copy()
    for i in r.choice(N, 20, replace=False):      # unsorted rows are legal
        r.shuffle(indices[indptr[i]:indptr[i + 1]])
    _assert_plan_equal(indptr, indices, T, C)


def test_plan_multi_edges_and_empty():
    _assert_plan_equal(np.array([0, 4, 4, 7], np.int32),
                       np.array([2, 1, 2, 2, 0, 0, 1], np.int32), 2, 2)
    _assert_plan_equal(np.zeros(9, np.int32), np.zeros(0, np.int32), 0, 0)


def test_plan_many_nodes_radix_passes():
    """N above 2^16 and 2^24 boundaries: three radix passes over source ids."""
    N = (1 << 17) + 3
    r = np.random.default_rng(9)
    deg = r.poisson(3.0, N)
    indptr = np.zeros(N + 1, np.int64)
    np.cumsum(deg, out=indptr[1:])
    indices = r.integers(0, N, int(indptr[-1])).astype(np.int32)   # multi-edges allowed
    _assert_plan_equal(indptr.astype(np.int32), indices, 8, 8)


@pytest.mark.parametrize("name", ["er1k", "powerlaw170k", "lognormal233k",
                                  "gatv2_powerlaw2m4", "sbm1m"])
def test_plan_workloads(name):
    indptr, indices = hp.workload_graph(name)
    info = _assert_plan_equal(indptr, indices, 0, 0)
    print(name, info)


@pytest.mark.parametrize("bad", ["index_high", "index_negative", "indptr_decreasing",
                                 "indptr_last", "indptr_first"])
def test_bad_graph_rejected(bad):
    indptr = np.array([0, 2, 3, 5], np.int32)
    indices = np.array([1, 2, 0, 0, 1], np.int32)
    if bad == "index_high":
        indices[3] = 3
    elif bad == "index_negative":
        indices[0] = -1
    elif bad == "indptr_decreasing":
        indptr[2] = 1
    elif bad == "indptr_last":
        indptr[3] = 4            # M = 5 edges but indptr[N] = 4
    elif bad == "indptr_first":
        indptr[0] = 1
    with pytest.raises(gb.GattnError) as ei:
        _plan_on_gpu(indptr, indices, 0, 0)
    assert ei.value.status == 2


def test_unsupported_and_invalid_args():
    indptr = np.array([0, 1, 2], np.int32)
    indices = np.array([1, 0], np.int32)
    plan = _plan_on_gpu(indptr, indices, 0, 0)
    try:
        dev = torch.device("cuda")
        for H, D, dt in ((3, 16, torch.bfloat16), (2, 4, torch.bfloat16), (2, 256, torch.float32),
                         (32, 64, torch.bfloat16)):
            with pytest.raises(gb.GattnError) as ei:
                gb.gattn_workspace_size(plan, H, D, dt)
            assert ei.value.status == 3
        Q = torch.zeros((2, 2, 16), device=dev)
        small = torch.empty(16, dtype=torch.uint8, device=dev)
        need = gb.gattn_workspace_size(plan, 2, 16, torch.float32)
        if need > 16:
            with pytest.raises(gb.GattnError) as ei:
                gb.gattn_fwd(plan, Q, Q, Q, gb.Score("dot"), workspace=small)
            assert ei.value.status == 1
        with pytest.raises(gb.GattnError) as ei:
            gb.gattn_fwd(plan, Q, Q, Q, gb.Score("gatv2", a=torch.zeros(0, device=dev)))
        assert ei.value.status == 1
    finally:
        plan.close()
