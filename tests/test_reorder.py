"""Node relabelling through the C ABI.

The host entry points (gattn_reorder, gattn_permute_csr) run without a GPU
and must equal the oracle's relabelling bit for bit; the device row
permutation and attention on a relabelled graph need the GPU."""
import numpy as np
import pytest

import oracle
from gnn_sparse_attention_gb300 import binding as gb
from gnn_sparse_attention_gb300 import build as gbuild
from gnn_sparse_attention_gb300 import synth


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    return gb.load_library()


def _graphs():
    yield synth.small_graph(0, 60, 3.0, isolated=0.1)
    yield synth.small_graph(1, 500, 1.2)
    yield synth.small_graph(2, 300, 8.0, hub_deg=250, self_loops=True)
    ip, ix = synth.small_graph(3, 200, 4.0)
    rows = [list(ix[ip[i]:ip[i + 1]]) for i in range(200)]
    rows[5] += rows[5][:3]                     # repeated sources
    ptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    yield ptr, np.array([j for r in rows for j in r], np.int32)
    yield np.zeros(1, np.int32), np.zeros(0, np.int32)           # empty graph


@pytest.mark.parametrize("kind,method", [("degree", oracle.REORDER_DEGREE),
                                         ("rcm", oracle.REORDER_RCM)])
def test_host_relabelling_matches_oracle(kind, method):
    for ip, ix in _graphs():
        perm = gb.gattn_reorder(ip, ix, kind)
        np.testing.assert_array_equal(perm, oracle.reorder(ip, ix, method))
        got = gb.gattn_permute_csr(ip, ix, perm)
        want = oracle.permute_csr(ip, ix, perm)
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_array_equal(got[1], want[1])


@pytest.mark.parametrize("kind,method", [("degree", oracle.REORDER_DEGREE),
                                         ("rcm", oracle.REORDER_RCM)])
def test_host_relabelling_powerlaw170k(kind, method):
    ip, ix = synth.make_graph(synth.WORKLOADS["powerlaw170k"])
    perm = gb.gattn_reorder(ip, ix, kind)
    np.testing.assert_array_equal(perm, oracle.reorder(ip, ix, method))


def test_host_relabelling_rejects_bad_input():
    ip, ix = synth.small_graph(4, 50, 3.0)
    with pytest.raises(gb.GattnError) as e:
        gb.gattn_permute_csr(ip, ix, np.zeros(50, np.int32))
    assert e.value.status == 1  # GATTN_ERR_INVALID_ARG
    bad = ix.copy()
    bad[0] = 50
    with pytest.raises(gb.GattnError) as e:
        gb.gattn_reorder(ip, bad, "rcm")
    assert e.value.status == 2  # GATTN_ERR_BAD_GRAPH
    with pytest.raises(KeyError):
        gb.gattn_reorder(ip, ix, "spectral")


# --------------------------------------------------------------------- GPU
torch = pytest.importorskip("torch")
needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@needs_gpu
@pytest.mark.gpu
def test_permute_rows_round_trip():
    r = np.random.default_rng(0)
    N = 1001
    perm = torch.from_numpy(r.permutation(N).astype(np.int32)).cuda()
    x = torch.randn(N, 4, 32, device="cuda").to(torch.bfloat16)
    y = gb.gattn_permute_rows(x, perm)
    assert torch.equal(y, x[perm.long()])
    z = gb.gattn_permute_rows(y, perm, inverse=True)
    torch.cuda.synchronize()
    assert torch.equal(z, x)


@needs_gpu
@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["degree", "rcm"])
def test_attention_on_relabelled_graph(kind):
    """Attention on the relabelled graph with relabelled features equals the
    relabelled attention of the original graph (and the oracle)."""
    from tests.helpers import TOL, GpuCase, compare, full_oracle
    ip, ix = synth.small_graph(7, 3000, 9.0, isolated=0.02, hub_deg=900)
    perm = gb.gattn_reorder(ip, ix, kind)
    ptr, idx = gb.gattn_permute_csr(ip, ix, perm)
    base = GpuCase(ip, ix, 4, 16, "bf16", "dot", seed=1)
    w = synth.Workload("t", "er", len(ip) - 1, 4, 16, "bf16", "dot")
    f = synth.make_features(w, seed=1)
    feats = {k: v[perm] for k, v in f.items() if k != "a"}
    rel = GpuCase(ptr, idx, 4, 16, "bf16", "dot", feats=feats)
    try:
        a, b = base.run(), rel.run()
        pt = torch.from_numpy(perm).cuda()
        for k in ("out", "dQ", "dK", "dV"):
            back = gb.gattn_permute_rows(b[k], pt, inverse=True)
            torch.cuda.synchronize()
            diff = (back.double() - a[k].double()).abs().max().item()
            assert diff <= TOL["bf16"] * a[k].double().abs().max().item(), k
        compare(b, full_oracle(rel), TOL["bf16"])
    finally:
        base.close()
        rel.close()
