"""The bounded-wait failure path of the attention passes, run on purpose.

Every wait of the gather pipeline has an iteration limit; on expiry a warp
records the failure in the plan, waits (bounded, with the normal limit) for
the copies it already issued, and returns, and gattn_plan_check_errors
reports GATTN_ERR_TIMEOUT.  gattn_plan_set_wait_test makes every warp's
first wait expire without polling, so that path runs without any wait that
never completes: the test checks that each pass reports the timeout, that
nothing is left in flight (the context stays usable and the error is not
sticky), and that the same plan gives the oracle's results once the hook is
cleared.
"""
import pytest

from tests import helpers as hp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gnn_sparse_attention_gb300 import binding as gb  # noqa: E402

TIMEOUT = 6


def _expect_timeout(plan):
    with pytest.raises(gb.GattnError) as ei:
        gb.gattn_plan_check_errors(plan)
    assert ei.value.status == TIMEOUT
    gb.gattn_plan_check_errors(plan)  # the record was cleared


@pytest.mark.parametrize("kind,dtype", [("dot", "f32"), ("gatv2", "bf16")])
def test_wait_timeout_is_reported_and_the_plan_recovers(kind, dtype):
    # hub destinations and a hub source with threshold/chunk 16: heavy chunks
    # and merge trees in both passes
    indptr, indices = hp.graph_with_source_hub(31, 900, 12.0, isolated=0.05, hub_deg=700)
    case = hp.GpuCase(indptr, indices, 4, 16, dtype, kind, seed=8, T=16, C=16)
    try:
        info = case.plan.info()
        assert info["n_chunks"] > 10 and info["n_src_chunks"] > 10
        Q, K, V, G = (case.t[k] for k in ("Q", "K", "V", "dO"))
        gb.gattn_plan_set_wait_test(case.plan, True)
        out, lse = gb.gattn_fwd(case.plan, Q, K, V, case.score)
        torch.cuda.synchronize()
        _expect_timeout(case.plan)
        # out / lse are undefined after a timeout: make valid ones for the
        # backward passes with the hook off, then turn it on again
        gb.gattn_plan_set_wait_test(case.plan, False)
        out, lse = gb.gattn_fwd(case.plan, Q, K, V, case.score)
        gb.gattn_plan_check_errors(case.plan)
        gb.gattn_plan_set_wait_test(case.plan, True)
        gb.gattn_bwd_dq(case.plan, Q, K, V, out, G, lse, case.score)
        torch.cuda.synchronize()
        _expect_timeout(case.plan)
        gb.gattn_bwd_dkdv(case.plan, Q, K, V, G, lse, case.score)
        torch.cuda.synchronize()
        _expect_timeout(case.plan)
        out_n = torch.empty_like(Q)
        lse_n = torch.empty_like(lse)
        gb.gattn_fwd_noalloc(case.plan, Q, K, V, case.score, out_n, lse_n)
        torch.cuda.synchronize()
        _expect_timeout(case.plan)
        # hook off: the same plan is whole again (counters cleared) and the
        # context still runs other work
        gb.gattn_plan_set_wait_test(case.plan, False)
        assert float(torch.ones(1 << 20, device=Q.device).sum()) == float(1 << 20)
        for _ in range(2):
            got = case.run()
            hp.compare(got, hp.full_oracle(case), hp.TOL[dtype])
    finally:
        case.close()
