"""Dense-tile path on the GPU through the C ABI: the device-built tile split
is bit-exact against the oracle's; the forward and the backward that run the
tiles on the tensor cores (plus the residual CSR / CSC passes) match the
oracle's softmax attention and its analytic gradients, and agree with the
CSR-only path of an untiled plan."""
import numpy as np
import pytest

import oracle
from gnn_sparse_attention_gb300 import synth
from tests.helpers import TOL, GpuCase, compare, full_oracle, relerr, sampled_oracle, to64

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

pytestmark = pytest.mark.gpu


def sbm_graph(N, p_in=0.5, inter=4, seed=0, block=64):
    w = synth.Workload("sbm_case", "sbm", N, 1, 64, "bf16", "dot", False,
                       {"block": block, "p_in": p_in, "inter_per_node": inter})
    return synth.make_graph(w, seed=seed)


def with_extras(indptr, indices, seed, dup=40, isolate=0.05):
    """Repeat some edges (multi-edges inside dense blocks), empty some rows,
    shuffle every row's order."""
    r = np.random.default_rng(seed)
    N = len(indptr) - 1
    rows = [list(indices[indptr[i]:indptr[i + 1]]) for i in range(N)]
    for _ in range(dup):
        i = int(r.integers(N))
        if rows[i]:
            rows[i].append(rows[i][int(r.integers(len(rows[i])))])
    for i in range(N):
        if r.random() < isolate:
            rows[i] = []
        r.shuffle(rows[i])
    ptr = np.zeros(N + 1, np.int64)
    ptr[1:] = np.cumsum([len(x) for x in rows])
    return ptr.astype(np.int32), np.array([j for x in rows for j in x], np.int32)


def dense_blocks_graph(N, pairs, p, seed, extra=2):
    """Edges j -> i kept with probability p inside the listed (row block,
    column block) pairs of 128 ids, plus ``extra`` uniform in-edges per node
    (repeats allowed): several tiles per row block and per column block."""
    r = np.random.default_rng(seed)
    rows = [[] for _ in range(N)]
    for rb, cb in pairs:
        j0, j1 = cb * 128, min(cb * 128 + 128, N)
        for i in range(rb * 128, min(rb * 128 + 128, N)):
            rows[i].extend((np.nonzero(r.random(j1 - j0) < p)[0] + j0).tolist())
    for i in range(N):
        rows[i].extend(r.integers(0, N, extra).tolist())
        r.shuffle(rows[i])
    ptr = np.zeros(N + 1, np.int64)
    ptr[1:] = np.cumsum([len(x) for x in rows])
    return ptr.astype(np.int32), np.array([j for x in rows for j in x], np.int32)


def export_tiles(case):
    from gnn_sparse_attention_gb300 import binding as gb
    return gb.gattn_plan_export_tiles(case.plan)


@pytest.mark.parametrize("N,density,extras", [(1000, 0.0625, False), (2048, 0.2, True),
                                              (640, 1e-4, True), (300, 1.0, False)])
def test_tile_split_matches_oracle(N, density, extras):
    ip, ix = sbm_graph(N, seed=N)
    if extras:
        ip, ix = with_extras(ip, ix, seed=N)
    case = GpuCase(ip, ix, 1, 64, "bf16", "dot", tile=True, density=density)
    try:
        got = export_tiles(case)
        info = case.plan.info()
        want = oracle.tile_plan(ip, ix, oracle.tile_min_count(density))
        assert info["tile_min_edges"] == oracle.tile_min_count(density)
        for k in ("tile_rb", "tile_cb", "masks", "indptr_r", "indices_r"):
            np.testing.assert_array_equal(got[k], want[k], err_msg=k)
        assert info["n_tiles"] == len(want["tile_rb"])
        assert info["n_tile_rows"] == len(np.unique(want["tile_rb"]))
    finally:
        case.close()


@pytest.mark.parametrize("N,H,D,extras", [(1000, 2, 64, False), (777, 1, 128, True),
                                          (1024, 4, 64, True), (130, 2, 64, False)])
def test_tile_forward_and_backward_parity(N, H, D, extras):
    ip, ix = sbm_graph(N, seed=N + 1)
    if extras:
        ip, ix = with_extras(ip, ix, seed=N + 1)
    case = GpuCase(ip, ix, H, D, "bf16", "dot", seed=3, tile=True)
    try:
        assert case.plan.info()["n_tiles"] > 0
        compare(case.run(), full_oracle(case), TOL["bf16"])
    finally:
        case.close()


def test_tile_and_csr_forward_agree():
    ip, ix = with_extras(*sbm_graph(1500, seed=9), seed=9)
    from gnn_sparse_attention_gb300 import binding as gb
    a = GpuCase(ip, ix, 2, 64, "bf16", "dot", seed=5, tile=True)
    b = GpuCase(ip, ix, 2, 64, "bf16", "dot", seed=5)
    try:
        oa, la = gb.gattn_fwd(a.plan, a.t["Q"], a.t["K"], a.t["V"], a.score)
        ob, lb = gb.gattn_fwd(b.plan, b.t["Q"], b.t["K"], b.t["V"], b.score)
        torch.cuda.synchronize()
        la, lb = to64(la), to64(lb)
        assert np.array_equal(np.isneginf(la), np.isneginf(lb))
        fin = np.isfinite(lb)
        # both sum fp32 weights; the orders differ (tile MMA vs CSR stream)
        assert np.abs(la[fin] - lb[fin]).max() < 1e-4
        assert relerr(to64(oa), to64(ob)) < TOL["bf16"]
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("dtype,kind,D", [("f32", "dot", 64), ("bf16", "gatv2", 64),
                                          ("bf16", "dot", 32)])
def test_tile_plan_other_layouts_use_the_csr_pass(dtype, kind, D):
    ip, ix = sbm_graph(700, seed=4)
    case = GpuCase(ip, ix, 2, D, dtype, kind, seed=6, tile=True)
    try:
        compare(case.run(), full_oracle(case), TOL[dtype])
    finally:
        case.close()


def test_tile_forward_is_deterministic():
    ip, ix = sbm_graph(1024, seed=12)
    from gnn_sparse_attention_gb300 import binding as gb
    case = GpuCase(ip, ix, 2, 64, "bf16", "dot", seed=1, tile=True)
    try:
        o1, l1 = gb.gattn_fwd(case.plan, case.t["Q"], case.t["K"], case.t["V"], case.score)
        o2, l2 = gb.gattn_fwd(case.plan, case.t["Q"], case.t["K"], case.t["V"], case.score)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    finally:
        case.close()


@pytest.mark.slow
def test_sbm1m_tiles_full_size():
    """The SBM workload (N = 2^20, 64-node communities, H = 8, D = 64, bf16) with
    the default tile density: every 128-node row block holds one diagonal tile;
    the split is bit-exact and sampled rows match the oracle."""
    w = synth.WORKLOADS["sbm1m"]
    ip, ix = synth.make_graph(w, seed=0)
    feats = synth.make_features(w, seed=0)
    case = GpuCase(ip, ix, w.H, w.D, w.dtype, w.score, feats=feats, tile=True)
    try:
        info = case.plan.info()
        assert info["n_tile_rows"] == (1 << 20) // 128
        got = export_tiles(case)
        want = oracle.tile_plan(ip, ix, info["tile_min_edges"])
        for k in ("tile_rb", "tile_cb", "masks", "indptr_r", "indices_r"):
            np.testing.assert_array_equal(got[k], want[k], err_msg=k)
        res = case.run()
        r = np.random.default_rng(0)
        rows = np.unique(np.concatenate([r.integers(0, w.N, 200), [0, 127, 128, w.N - 1]]))
        srcs = np.unique(r.integers(0, w.N, 50))
        ref = sampled_oracle(case, rows, srcs)
        compare({k: res[k] for k in ("out", "lse", "dQ")}, ref["rows"], TOL["bf16"], rows=rows)
        compare({k: res[k] for k in ("dK", "dV")}, ref["srcs"], TOL["bf16"], rows=srcs)
    finally:
        case.close()


BLOCK_PAIRS = [(0, 0), (0, 1), (0, 2), (1, 1), (2, 1), (2, 3), (3, 0), (4, 4), (4, 1)]


@pytest.mark.parametrize("H,D,p", [(2, 64, 0.3), (1, 128, 0.5), (4, 64, 0.08)])
def test_tile_backward_several_tiles_per_block(H, D, p):
    """Row blocks and column blocks with up to four tiles each (the gradient
    accumulators sum over a block's tiles), a partial last block, repeated
    edges and random residual edges: forward and backward against the oracle."""
    ip, ix = dense_blocks_graph(600, BLOCK_PAIRS, p, seed=int(p * 100) + D)
    case = GpuCase(ip, ix, H, D, "bf16", "dot", seed=7, tile=True)
    try:
        info = case.plan.info()
        want = oracle.tile_plan(ip, ix, info["tile_min_edges"])
        assert info["n_tiles"] == len(want["tile_rb"]) >= 7
        compare(case.run(), full_oracle(case), TOL["bf16"])
    finally:
        case.close()


def test_tile_and_csr_backward_agree():
    ip, ix = with_extras(*sbm_graph(1500, seed=19), seed=19)
    a = GpuCase(ip, ix, 2, 64, "bf16", "dot", seed=8, tile=True)
    b = GpuCase(ip, ix, 2, 64, "bf16", "dot", seed=8)
    try:
        ra, rb = a.run(), b.run()
        for k in ("dQ", "dK", "dV"):
            assert relerr(to64(ra[k]), to64(rb[k])) < TOL["bf16"], k
        ref = full_oracle(b)
        compare(ra, ref, TOL["bf16"])
        compare(rb, ref, TOL["bf16"])
    finally:
        a.close()
        b.close()


def test_tile_backward_is_deterministic():
    ip, ix = dense_blocks_graph(520, BLOCK_PAIRS[:6], 0.4, seed=3)
    from gnn_sparse_attention_gb300 import binding as gb
    case = GpuCase(ip, ix, 2, 64, "bf16", "dot", seed=2, tile=True)
    try:
        Q, K, V, G = (case.t[k] for k in ("Q", "K", "V", "dO"))
        out, lse = gb.gattn_fwd(case.plan, Q, K, V, case.score)
        g1 = gb.gattn_bwd(case.plan, Q, K, V, out, G, lse, case.score)
        g2 = gb.gattn_bwd(case.plan, Q, K, V, out, G, lse, case.score)
        torch.cuda.synchronize()
        gb.gattn_plan_check_errors(case.plan)
        for x, y in zip(g1[:3], g2[:3]):
            assert torch.equal(x, y)
    finally:
        case.close()


def _transposed_masks(masks):
    """masks [n, 128 rows, 4 words] -> [n, 128 columns, 4 words] (numpy bit transpose)."""
    bits = np.unpackbits(masks.view(np.uint8).reshape(len(masks), 128, 16), axis=2,
                         bitorder="little").reshape(len(masks), 128, 128)   # [t, row, column]
    return np.packbits(bits.transpose(0, 2, 1).reshape(len(masks), 128, 128), axis=2,
                       bitorder="little").reshape(len(masks), 128, 16).view(np.uint32)


@pytest.mark.parametrize("kind", ["sbm", "blocks", "blocks_sparse"])
def test_tile_backward_plan_matches_oracle(kind):
    """The residual CSC is the oracle plan's CSC of the oracle's residual CSR,
    the column grouping is a stable sort of the oracle's tiles by column
    block, and the transposed masks are the oracle's masks transposed."""
    from gnn_sparse_attention_gb300 import binding as gb
    if kind == "sbm":
        ip, ix = with_extras(*sbm_graph(1200, seed=21), seed=21)
    else:
        ip, ix = dense_blocks_graph(600, BLOCK_PAIRS, 0.3 if kind == "blocks" else 0.08, seed=5)
    case = GpuCase(ip, ix, 1, 64, "bf16", "dot", tile=True)
    try:
        got = gb.gattn_plan_export_tile_bwd(case.plan)
        info = case.plan.info()
        tp = oracle.tile_plan(ip, ix, info["tile_min_edges"])
        res = oracle.plan(tp["indptr_r"], tp["indices_r"], 32, 32)
        np.testing.assert_array_equal(got["indptrT_r"], res["indptrT"])
        np.testing.assert_array_equal(got["csc_dst_r"], res["csc_dst"])
        order = np.argsort(tp["tile_cb"], kind="stable").astype(np.int32)
        cbs, starts = np.unique(tp["tile_cb"][order], return_index=True)
        np.testing.assert_array_equal(got["tcol_tile"], order)
        np.testing.assert_array_equal(got["tcol_cb"], cbs)
        np.testing.assert_array_equal(got["tcol_ptr"], np.append(starts, len(order)))
        np.testing.assert_array_equal(got["masks_t"], _transposed_masks(tp["masks"]))
    finally:
        case.close()
