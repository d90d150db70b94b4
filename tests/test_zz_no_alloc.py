"""gattn_fwd_noalloc: the forward pass for callers that cannot allocate device
memory where they run the layer (code under an allocator or memory pool it
does not own, plugin hosts that hand over only the input and output
tensors).  Its scratch is a fixed array inside the library.  Through the C
ABI the tests check that two calls in a row give exactly gattn_fwd's result
on an untiled plan (both run the same deterministic kernel over the same
plan) and the oracle's result within the bf16 bar on a tiled plan, that the
call allocates nothing, that misaligned pointers and a plan needing more
scratch than the array holds are refused on the host.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest

from tests import helpers as hp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gnn_sparse_attention_gb300 import binding as gb  # noqa: E402
from gnn_sparse_attention_gb300 import synth  # noqa: E402


def _two_calls(case, check):
    """Run gattn_fwd_noalloc twice into poisoned outputs; check() each result."""
    Q, K, V = (case.t[k] for k in ("Q", "K", "V"))
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
            # the first call in a context looks up the library's fixed array
            # (its documented set-up); later calls take nothing
            assert torch.cuda.mem_get_info()[0] == free0
        gb.gattn_plan_check_errors(case.plan)
        check(out, lse)


@pytest.mark.parametrize("kind", ["dot", "gatv2"])
def test_fwd_noalloc_equals_fwd(kind):
    # hub destinations with threshold/chunk 16: many heavy chunks use the scratch
    indptr, indices = hp.graph_with_source_hub(21, 1500, 20.0, isolated=0.05, hub_deg=1200)
    case = hp.GpuCase(indptr, indices, 8, 16, "bf16", kind, seed=4, T=16, C=16)
    try:
        assert case.plan.info()["n_chunks"] > 100
        Q, K, V = (case.t[k] for k in ("Q", "K", "V"))
        ref_out, ref_lse = gb.gattn_fwd(case.plan, Q, K, V, case.score)
        torch.cuda.synchronize()

        def check(out, lse):
            assert torch.equal(out, ref_out)
            assert torch.equal(lse, ref_lse)   # -inf of isolated nodes included

        _two_calls(case, check)
    finally:
        case.close()


def test_fwd_noalloc_tiled_plan_matches_oracle():
    # a block-model graph whose 128-node blocks become tensor-core tiles in
    # gattn_fwd; the no-alloc call runs the CSR pass over every edge instead
    w = synth.Workload("sbm_case", "sbm", 1024, 2, 64, "bf16", "dot", False,
                       {"block": 64, "p_in": 0.5, "inter_per_node": 4})
    indptr, indices = synth.make_graph(w, seed=2)
    case = hp.GpuCase(indptr, indices, 2, 64, "bf16", "dot", seed=9, tile=True, T=32, C=32)
    try:
        assert case.plan.info()["n_tiles"] > 0 and case.plan.info()["n_chunks"] > 0
        ref = hp.full_oracle(case)

        def check(out, lse):
            hp.compare({"out": out, "lse": lse}, ref, hp.TOL["bf16"])

        _two_calls(case, check)
    finally:
        case.close()


def test_fwd_noalloc_rejects_misaligned_pointers():
    indptr, indices = synth.small_graph(3, 200, 6.0)
    for kind in ("dot", "gatv2"):
        case = hp.GpuCase(indptr, indices, 2, 16, "f32", kind, seed=2)
        try:
            lib = gb.load_library()
            Q, K, V = (case.t[k] for k in ("Q", "K", "V"))
            out = torch.empty_like(Q)
            raw = torch.empty(Q.shape[0] * 2 * 4 + 16, dtype=torch.uint8, device=Q.device)
            good_lse = raw.data_ptr()
            bad_lse = raw.data_ptr() + 2          # not 4-byte aligned
            sc = case.score._struct()

            def call(lse_ptr, score):
                return lib.gattn_fwd_noalloc(case.plan.handle, 2, 16, gb.GATTN_F32, Q.data_ptr(),
                                             K.data_ptr(), V.data_ptr(), ctypes.byref(score),
                                             out.data_ptr(), lse_ptr, None)

            assert call(bad_lse, sc) == 1
            assert b"lse" in lib.gattn_last_error()
            if kind == "gatv2":
                a_raw = torch.empty(2 * 16 * 4 + 16, dtype=torch.uint8, device=Q.device)
                sc_bad = case.score._struct()
                sc_bad.a = a_raw.data_ptr() + 2   # not 4-byte aligned
                assert call(good_lse, sc_bad) == 1
                assert b"a[H*D]" in lib.gattn_last_error()
            torch.cuda.synchronize()
            gb.gattn_plan_check_errors(case.plan)
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
