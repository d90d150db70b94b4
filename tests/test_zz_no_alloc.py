"""gattn_fwd_noalloc: the forward pass for callers that cannot allocate
device memory at call time (inside CUDA graph capture, under a memory pool
they do not own).  Its scratch is a fixed array inside the library; the test
checks, through the C ABI, that two calls in a row give the same result as
gattn_fwd with a caller workspace, that the call allocates nothing, and that
a plan needing more scratch than the array holds is refused.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

from tests import helpers as hp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gnn_sparse_attention_gb300 import binding as gb  # noqa: E402


@pytest.mark.parametrize("kind", ["dot", "gatv2"])
def test_fwd_noalloc_matches_fwd(kind):
    # hub destinations with threshold/chunk 16: many heavy chunks use the scratch
    indptr, indices = hp.graph_with_source_hub(21, 1500, 20.0, isolated=0.05, hub_deg=1200)
    case = hp.GpuCase(indptr, indices, 8, 16, "bf16", kind, seed=4, T=16, C=16)
    try:
        assert case.plan.info()["n_chunks"] > 100
        Q, K, V = (case.t[k] for k in ("Q", "K", "V"))
        ref_out, ref_lse = gb.gattn_fwd(case.plan, Q, K, V, case.score)
        torch.cuda.synchronize()
        out = torch.empty_like(Q)
        lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=Q.device)
        for call in range(2):
            out.fill_(7.0)
            lse.fill_(7.0)
            torch.cuda.synchronize()
            alloc0 = torch.cuda.memory_allocated()
            free0 = torch.cuda.mem_get_info()[0]
            gb.gattn_fwd_noalloc(case.plan, Q, K, V, case.score, out, lse)
            torch.cuda.synchronize()
            assert torch.cuda.memory_allocated() == alloc0
            if call > 0:
                # the first call on a device loads the library's fixed array
                # (its documented set-up); later calls take nothing
                assert torch.cuda.mem_get_info()[0] == free0
            gb.gattn_plan_check_errors(case.plan)
            assert hp.relerr(out.double().cpu().numpy(), ref_out.double().cpu().numpy()) <= 2e-2
            fin = torch.isfinite(ref_lse)
            assert torch.equal(torch.isfinite(lse), fin)
            assert hp.relerr(lse[fin].double().cpu().numpy(), ref_lse[fin].double().cpu().numpy()) <= 2e-2
    finally:
        case.close()


def test_fwd_noalloc_rejects_oversized_scratch():
    # 5000 nodes of degree 64 in chunks of 16 with 1 KB rows: ~53 MB of partials
    N, deg = 5000, 64
    r = np.random.default_rng(3)
    rows = [np.sort(r.choice(np.setdiff1d(np.arange(N), [i]), deg, replace=False))
            for i in range(N)]
    indptr = (np.arange(N + 1) * deg).astype(np.int32)
    indices = np.concatenate(rows).astype(np.int32)
    case = hp.GpuCase(indptr, indices, 8, 64, "bf16", "dot", seed=1, T=16, C=16)
    try:
        Q, K, V = (case.t[k] for k in ("Q", "K", "V"))
        out = torch.empty_like(Q)
        lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=Q.device)
        with pytest.raises(gb.GattnError) as ei:
            gb.gattn_fwd_noalloc(case.plan, Q, K, V, case.score, out, lse)
        assert ei.value.status == 1
        assert "scratch" in str(ei.value)
    finally:
        case.close()
