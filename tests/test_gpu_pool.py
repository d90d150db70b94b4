"""Max / min pooling on the GPU through the C ABI against the oracle: the
forward is exact (values and smallest-id argmax, bit for bit), the backward
within the dtype's tolerance; heavy nodes (edge chunks merged by packed
atomics), ties, isolated nodes and both dtypes are covered."""
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


def _run(ip, ix, X, dtype, op, T=0, C=0, G=None):
    dev = torch.device("cuda")
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    plan = gb.gattn_plan_create(torch.from_numpy(ip).to(dev), torch.from_numpy(ix).to(dev), T, C)
    try:
        x = torch.from_numpy(np.ascontiguousarray(X, np.float32)).to(dev, tdt)
        out, arg = gb.gattn_pool_fwd(plan, x, op)
        res = {"out": out.double().cpu().numpy(), "arg": arg.cpu().numpy(),
               "x64": x.double().cpu().numpy()}
        if G is not None:
            g = torch.from_numpy(np.ascontiguousarray(G, np.float32)).to(dev, tdt)
            dx = gb.gattn_pool_bwd(plan, arg, g)
            res["dx"] = dx.double().cpu().numpy()
            res["g64"] = g.double().cpu().numpy()
        torch.cuda.synchronize()
        gb.gattn_plan_check_errors(plan)
        return res
    finally:
        plan.close()


@pytest.mark.parametrize("dtype,F", [("bf16", 16), ("bf16", 128), ("bf16", 1024), ("f32", 8),
                                     ("f32", 64), ("f32", 512)])
@pytest.mark.parametrize("op", ["max", "min"])
def test_pool_matches_oracle(dtype, F, op):
    ip, ix = synth.small_graph(21, 900, 7.0, isolated=0.08, hub_deg=700)
    r = np.random.default_rng(F)
    X = r.standard_normal((900, F))
    X[::7] = np.round(X[::7] * 2) / 2          # coarse values: many ties across sources
    G = r.standard_normal((900, F))
    got = _run(ip, ix, X, dtype, op, T=16, C=16, G=G)
    o = oracle.MAX if op == "max" else oracle.MIN
    out, arg = oracle.reduce_forward(ip, ix, got["x64"], o)
    np.testing.assert_array_equal(got["out"], out)
    np.testing.assert_array_equal(got["arg"], arg)
    dx = oracle.reduce_backward(arg, got["g64"], 900)
    assert relerr(got["dx"], dx) <= TOL[dtype]


def test_pool_all_ties_and_repeated_edges():
    # every source holds the same row: arg must be each node's smallest source
    ip, ix = synth.small_graph(22, 400, 30.0, hub_deg=390)
    rows = [list(ix[ip[i]:ip[i + 1]]) for i in range(400)]
    rows[-1] += list(ix[:50])                                   # repeated edges into the last row
    ip2 = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    ix2 = np.array([j for x in rows for j in x], np.int32)
    X = np.ones((400, 32))
    got = _run(ip2, ix2, X, "bf16", "max", T=32, C=32)
    out, arg = oracle.reduce_forward(ip2, ix2, got["x64"], oracle.MAX)
    np.testing.assert_array_equal(got["out"], out)
    np.testing.assert_array_equal(got["arg"], arg)


def test_pool_powerlaw170k_full():
    """The power-law workload's graph with F = 128 bf16 features (H*D of the
    attention workload), default plan: exact against the oracle."""
    w = synth.WORKLOADS["powerlaw170k"]
    ip, ix = synth.make_graph(w, seed=0)
    X = synth.normal(0, 1, (w.N, w.H * w.D))
    got = _run(ip, ix, X, "bf16", "max")
    out, arg = oracle.reduce_forward(ip, ix, got["x64"], oracle.MAX)
    np.testing.assert_array_equal(got["out"], out)
    np.testing.assert_array_equal(got["arg"], arg)


def test_pool_is_deterministic_and_reusable():
    ip, ix = synth.small_graph(23, 2000, 12.0, hub_deg=1500)
    X = np.random.default_rng(0).standard_normal((2000, 64))
    a = _run(ip, ix, X, "f32", "min", T=32, C=32)
    b = _run(ip, ix, X, "f32", "min", T=32, C=32)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["arg"], b["arg"])
