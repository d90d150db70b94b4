"""GATv2 on the GPU with LeakyReLU slopes other than 0.2 and with scores
whose pre-activation z = xl_i + xr_j is exactly zero.

The kernels evaluate LeakyReLU_s(z) as c1 z + c2 |z| (c1 = (1 + s) / 2,
c2 = (1 - s) / 2) in the forward and the CSC pass, and the source gradient
as a (s sum ds + (1 - s) sum_{z > 0} ds); the derivative at z = 0 is the
slope, as in the oracle.  Self-loops with xr = -xl make every element of
z_ii exactly zero (bf16 and fp32 alike), so that rule decides dXl and dXr
on those edges.
"""
import numpy as np
import pytest

import oracle
from tests import helpers as hp
from gnn_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _with_self_loops(indptr, indices):
    N = len(indptr) - 1
    rows = [sorted(set(indices[indptr[i]:indptr[i + 1]].tolist()) | {i}) for i in range(N)]
    ptr = np.zeros(N + 1, np.int64)
    ptr[1:] = np.cumsum([len(r) for r in rows])
    return ptr.astype(np.int32), np.array([j for r in rows for j in r], np.int32)


@pytest.mark.parametrize("slope", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("dtype,H,D", [("f32", 2, 16), ("bf16", 4, 32), ("bf16", 8, 64)])
def test_gatv2_slopes_and_zero_preactivation(slope, dtype, H, D):
    from gnn_sparse_attention_gb300 import binding as gb
    indptr, indices = hp.graph_with_source_hub(8, 500, 12.0, isolated=0.03, hub_deg=300)
    indptr, indices = _with_self_loops(indptr, indices)
    N = len(indptr) - 1
    w = synth.Workload("case", "er", N, H, D, dtype, "gatv2")
    f = synth.make_features(w, seed=21)
    f["K"] = -f["Q"]                      # z_ii = xl_i + xr_i = 0 on every self-loop
    tdt = hp.torch_dtype(dtype)
    dev = torch.device("cuda")
    t = {k: torch.from_numpy(np.ascontiguousarray(f[k])).to(dev, tdt) for k in ("Q", "K", "V", "dO")}
    a = torch.from_numpy(f["a"]).to(dev)
    score = gb.Score("gatv2", a=a, neg_slope=slope)
    plan = gb.gattn_plan_create(torch.from_numpy(indptr).to(dev),
                                torch.from_numpy(indices).to(dev), 16, 16)
    try:
        out, lse = gb.gattn_fwd(plan, t["Q"], t["K"], t["V"], score)
        dQ, dK, dV, da = gb.gattn_bwd(plan, t["Q"], t["K"], t["V"], out, t["dO"], lse, score)
        torch.cuda.synchronize()
        gb.gattn_plan_check_errors(plan)
        h = {k: t[k].double().cpu().numpy() for k in t}
        assert np.array_equal(h["K"], -h["Q"])
        r_out, r_lse = oracle.forward(indptr, indices, h["Q"], h["K"], h["V"], kind=oracle.GATV2,
                                      a=f["a"], slope=slope)
        r = oracle.backward(indptr, indices, h["Q"], h["K"], h["V"], h["dO"], kind=oracle.GATV2,
                            a=f["a"], slope=slope)
        hp.compare({"out": out, "lse": lse, "dQ": dQ, "dK": dK, "dV": dV, "da": da},
                   {"out": r_out, "lse": r_lse, "dQ": r[0], "dK": r[1], "dV": r[2], "da": r[3]},
                   hp.TOL[dtype])
    finally:
        plan.close()
