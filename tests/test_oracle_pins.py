"""Pins of the fp64 oracle to things other than itself (CPU only).

Each check is chosen so that a plausible slip in the oracle (a dropped scale,
a wrong softmax axis, a transposed edge direction, a sign error in the
softmax Jacobian, a missing LeakyReLU slope in a derivative, an unstable CSC
order) fails at least one of them:

* hand-worked closed-form examples (tests/golden/*_worked_example.json);
* dense masked softmax attention by brute force (N <= 64) with scipy's
  softmax / logsumexp -- a different formulation (dense N x N score matrix,
  -inf mask) from the oracle's sparse loops;
* closed forms: Q = 0 or a = 0 gives the neighbour mean, V = 1 gives 1
  (weights sum to one), degree one gives v_j, degree zero gives 0 / -inf;
* central finite differences of L = sum(G * out) for dQ, dK, dV, da;
* permutation equivariance under node relabelling;
* the plan against an independent recount (numpy stable sort, scipy CSC).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.sparse as sp
from scipy.special import logsumexp, softmax

import oracle
from gnn_sparse_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _closed(x):
    """Evaluate a closed-form expression string of a golden fixture."""
    env = {"sqrt": math.sqrt, "log": math.log, "inf": math.inf, "__builtins__": {}}
    if isinstance(x, list):
        return [_closed(v) for v in x]
    return float(eval(x, env))  # fixture strings are plain arithmetic expressions


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    arr = {k: np.array(_closed(g[k]), np.float64)
           for k in ("Q", "K", "V", "dO", "out", "lse", "dQ", "dK", "dV", "a") if k in g}
    return g, arr


def _graph(seed, N, avg, **kw):
    return synth.small_graph(seed, N, avg, **kw)


def _feats(seed, N, H, D):
    r = np.random.default_rng(seed + 1000)
    return [r.standard_normal((N, H, D)) for _ in range(4)]


# ----------------------------------------------------------------------------
# hand-worked examples
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name,kind", [("dot_worked_example.json", oracle.DOT),
                                       ("gatv2_worked_example.json", oracle.GATV2)])
def test_worked_example(name, kind):
    g, x = _load_golden(name)
    a = x.get("a")
    out, lse = oracle.forward(g["indptr"], g["indices"], x["Q"], x["K"], x["V"], kind=kind, a=a)
    np.testing.assert_allclose(out, x["out"], rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(x["lse"]))
    fin = np.isfinite(x["lse"])
    np.testing.assert_allclose(lse[fin], x["lse"][fin], rtol=0, atol=1e-13)
    dQ, dK, dV, da = oracle.backward(g["indptr"], g["indices"], x["Q"], x["K"], x["V"], x["dO"],
                                     kind=kind, a=a)
    np.testing.assert_allclose(dQ, x["dQ"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dK, x["dK"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dV, x["dV"], rtol=0, atol=1e-13)
    if kind == oracle.GATV2:
        np.testing.assert_allclose(da, np.array(_closed(g["da"])), rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------
# dense brute force
# ----------------------------------------------------------------------------
def _dense_attention(indptr, indices, Q, K, V, kind, a=None, slope=0.2):
    """Dense masked softmax attention: S[h, i, j] over all pairs, -inf off-graph."""
    N, H, D = Q.shape
    A = sp.csr_matrix((np.ones(len(indices)), np.asarray(indices), np.asarray(indptr)),
                      shape=(N, N)).toarray() > 0                     # A[i, j]: edge j -> i
    if kind == oracle.DOT:
        S = np.einsum("ihd,jhd->hij", Q, K) / math.sqrt(D)
    else:
        Z = Q[:, None, :, :] + K[None, :, :, :]                      # [i, j, h, d]
        S = np.einsum("ijhd,hd->hij", np.where(Z > 0, Z, slope * Z), a)
    S = np.where(A[None], S, -np.inf)
    has = A.any(axis=1)
    P = np.zeros_like(S)
    P[:, has] = softmax(S[:, has], axis=-1)
    out = np.einsum("hij,jhd->ihd", P, V)
    lse = np.full((N, H), -np.inf)
    lse[has] = logsumexp(S[:, has], axis=-1).T
    return out, lse


@pytest.mark.parametrize("kind", [oracle.DOT, oracle.GATV2])
@pytest.mark.parametrize("seed,N,H,D", [(1, 24, 2, 4), (2, 64, 3, 8), (3, 40, 1, 16)])
def test_dense_bruteforce(kind, seed, N, H, D):
    indptr, indices = _graph(seed, N, 6.0, isolated=0.1, hub_deg=N // 2)
    Q, K, V, _ = _feats(seed, N, H, D)
    a = np.random.default_rng(seed).standard_normal((H, D)) / math.sqrt(D)
    out, lse = oracle.forward(indptr, indices, Q, K, V, kind=kind, a=a)
    ref_out, ref_lse = _dense_attention(indptr, indices, Q, K, V, kind, a)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(ref_lse))
    np.testing.assert_allclose(lse[np.isfinite(lse)], ref_lse[np.isfinite(ref_lse)], atol=1e-12)


# ----------------------------------------------------------------------------
# closed forms and invariants
# ----------------------------------------------------------------------------
def test_equal_scores_give_neighbour_mean():
    N, H, D = 50, 2, 8
    indptr, indices = _graph(4, N, 5.0, isolated=0.1)
    _, K, V, _ = _feats(4, N, H, D)
    deg = np.diff(indptr)
    mean = np.zeros((N, H, D))
    for i in range(N):
        if deg[i]:
            mean[i] = V[indices[indptr[i]:indptr[i + 1]]].mean(axis=0)
    out, lse = oracle.forward(indptr, indices, np.zeros((N, H, D)), K, V)
    np.testing.assert_allclose(out, mean, atol=1e-13)
    np.testing.assert_allclose(lse[deg > 0], np.log(deg[deg > 0])[:, None].repeat(H, 1), atol=1e-13)
    out, _ = oracle.forward(indptr, indices, K, K, V, kind=oracle.GATV2, a=np.zeros((H, D)))
    np.testing.assert_allclose(out, mean, atol=1e-13)


def test_weights_sum_to_one_and_isolated_zero():
    N, H, D = 60, 4, 4
    indptr, indices = _graph(5, N, 7.0, isolated=0.2)
    Q, K, _, _ = _feats(5, N, H, D)
    deg = np.diff(indptr)
    out, lse = oracle.forward(indptr, indices, Q, K, np.ones((N, H, D)))
    np.testing.assert_allclose(out[deg > 0], 1.0, atol=1e-13)
    assert (out[deg == 0] == 0).all()
    assert np.isneginf(lse[deg == 0]).all()


def test_single_in_edge_copies_value():
    N, H, D = 30, 2, 4
    r = np.random.default_rng(6)
    src = np.array([(i + 1 + r.integers(0, N - 1)) % N for i in range(N)], np.int32)
    indptr = np.arange(N + 1, dtype=np.int32)
    Q, K, V, _ = _feats(6, N, H, D)
    out, lse = oracle.forward(indptr, src, Q, K, V)
    np.testing.assert_allclose(out, V[src], atol=1e-14)
    np.testing.assert_allclose(lse, np.einsum("ihd,ihd->ih", Q, K[src]) / 2.0, atol=1e-13)


@pytest.mark.parametrize("kind", [oracle.DOT, oracle.GATV2])
def test_permutation_equivariance(kind):
    N, H, D = 48, 2, 8
    indptr, indices = _graph(7, N, 6.0, isolated=0.1)
    Q, K, V, G = _feats(7, N, H, D)
    a = np.random.default_rng(7).standard_normal((H, D)) / math.sqrt(D)
    pi = np.random.default_rng(8).permutation(N)            # old id -> new id
    inv = np.argsort(pi)
    deg = np.diff(indptr)
    # relabelled graph: new row pi[i] holds sources pi[j]
    new_deg = deg[inv]
    new_ptr = np.zeros(N + 1, np.int64)
    np.cumsum(new_deg, out=new_ptr[1:])
    new_idx = np.concatenate([np.sort(pi[indices[indptr[o]:indptr[o + 1]]]) for o in inv])
    Pq, Pk, Pv, Pg = (X[inv] for X in (Q, K, V, G))
    out, lse = oracle.forward(indptr, indices, Q, K, V, kind=kind, a=a)
    pout, plse = oracle.forward(new_ptr, new_idx, Pq, Pk, Pv, kind=kind, a=a)
    np.testing.assert_allclose(pout, out[inv], atol=1e-12)
    np.testing.assert_allclose(plse, lse[inv], atol=1e-12)
    g = oracle.backward(indptr, indices, Q, K, V, G, kind=kind, a=a)
    pg = oracle.backward(new_ptr, new_idx, Pq, Pk, Pv, Pg, kind=kind, a=a)
    for x, px in zip(g[:3], pg[:3]):
        np.testing.assert_allclose(px, x[inv], atol=1e-12)
    if kind == oracle.GATV2:
        np.testing.assert_allclose(pg[3], g[3], atol=1e-12)


# ----------------------------------------------------------------------------
# finite differences
# ----------------------------------------------------------------------------
def _loss(indptr, indices, Q, K, V, G, kind, a):
    out, _ = oracle.forward(indptr, indices, Q, K, V, kind=kind, a=a)
    return float((out * G).sum())


@pytest.mark.parametrize("kind", [oracle.DOT, oracle.GATV2])
def test_finite_differences(kind):
    N, H, D = 20, 2, 3
    indptr, indices = _graph(9, N, 4.0, isolated=0.1, hub_deg=12)
    Q, K, V, G = _feats(9, N, H, D)
    a = np.random.default_rng(9).standard_normal((H, D))
    dQ, dK, dV, da = oracle.backward(indptr, indices, Q, K, V, G, kind=kind, a=a)
    h = 1e-6
    rows = np.repeat(np.arange(N), np.diff(indptr))

    def near_kink(name, idx):
        if kind != oracle.GATV2 or name not in ("Q", "K"):
            return False
        n, hh, d = idx
        e = rows == n if name == "Q" else indices == n
        z = Q[rows[e], hh, d] + K[indices[e], hh, d]
        return bool((np.abs(z) < 1e-3).any())

    tensors = {"Q": (Q, dQ), "K": (K, dK), "V": (V, dV)}
    if kind == oracle.GATV2:
        tensors["a"] = (a, da)
    checked = 0
    for name, (X, dX) in tensors.items():
        for idx in np.ndindex(X.shape):
            if near_kink(name, idx):
                continue
            old = X[idx]
            X[idx] = old + h
            lp = _loss(indptr, indices, Q, K, V, G, kind, a)
            X[idx] = old - h
            lm = _loss(indptr, indices, Q, K, V, G, kind, a)
            X[idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - dX[idx]) <= 1e-6 * max(1.0, abs(dX[idx])), (name, idx, fd, dX[idx])
            checked += 1
    assert checked > 3 * N * H * D * 0.9


@pytest.mark.parametrize("slope", [0.0, 0.2, 0.5])
def test_leaky_derivative_at_zero_takes_the_slope(slope):
    """The pages fix no derivative of LeakyReLU at its kink; the reading is
    LReLU'(0) = slope.  With x_r = -x_l every self-loop has z = 0 exactly.
    Moving x_l[i] down puts that edge on the linear side of slope s, so a
    left finite difference must equal the analytic gradient there, and a
    right one (which sees slope 1) must not."""
    N, H, D = 6, 2, 3
    indptr, indices = _graph(31, N, 3.0, self_loops=True)
    Q, K, V, G = _feats(31, N, H, D)
    K = -Q
    a = np.random.default_rng(31).standard_normal((H, D))
    dQ = oracle.backward(indptr, indices, Q, K, V, G, kind=oracle.GATV2, a=a, slope=slope)[0]

    def loss(Qx):
        out, _ = oracle.forward(indptr, indices, Qx, K, V, kind=oracle.GATV2, a=a, slope=slope)
        return float((out * G).sum())

    h = 1e-7
    L0 = loss(Q)
    far = 0.0
    for idx in np.ndindex(Q.shape):
        Qx = Q.copy()
        Qx[idx] -= h
        left = (L0 - loss(Qx)) / h
        Qx[idx] += 2 * h
        right = (loss(Qx) - L0) / h
        assert abs(left - dQ[idx]) <= 1e-5 * max(1.0, abs(dQ[idx])), (idx, left, dQ[idx])
        far = max(far, abs(right - dQ[idx]))
    assert far > 1e-3  # the right side sees slope 1: the kink convention is observable


# ----------------------------------------------------------------------------
# plan
# ----------------------------------------------------------------------------
def _plan_recount(indptr, indices, T, C):
    indptr = np.asarray(indptr, np.int64)
    indices = np.asarray(indices, np.int64)
    N = len(indptr) - 1
    M = int(indptr[-1])
    deg = np.diff(indptr)
    rows = np.repeat(np.arange(N), deg)
    eid = np.arange(M)
    order = np.lexsort((eid, indices))                   # by source, then edge id
    outdeg = np.bincount(indices, minlength=N)
    indptrT = np.concatenate([[0], np.cumsum(outdeg)])
    # scipy's CSR -> CSC conversion as a second, independent transpose
    csc = sp.csr_matrix((np.ones(M), indices, indptr), shape=(N, N)).tocsc()
    csc.sort_indices()
    assert (csc.indptr == indptrT).all()
    assert (csc.indices == rows[order]).all()

    def chunks_of(ptr, d):
        out = []
        for i in np.nonzero(d > T)[0]:
            for s in range(ptr[i], ptr[i + 1], C):
                out.append((i, s, min(s + C, ptr[i + 1])))
        return np.array(out, np.int64).reshape(-1, 3)

    def hist(d):
        b = np.where(d > 0, np.floor(np.log2(np.maximum(d, 1))) + 1, 0).astype(np.int64)
        return np.bincount(b, minlength=33)

    return {
        "deg": deg, "hist": hist(deg), "light": np.nonzero(deg <= T)[0],
        "chunks": chunks_of(indptr, deg), "indptrT": indptrT, "csc_dst": rows[order],
        "csc_eid": order, "outdeg": outdeg, "hist_out": hist(outdeg),
        "light_src": np.nonzero(outdeg <= T)[0], "src_chunks": chunks_of(indptrT, outdeg),
    }


@pytest.mark.parametrize("seed,N,avg,T,C", [(10, 200, 6.0, 8, 4), (11, 500, 20.0, 32, 16),
                                            (12, 64, 3.0, 0, 1), (13, 300, 10.0, 1000, 7)])
def test_plan_recount(seed, N, avg, T, C):
    indptr, indices = _graph(seed, N, avg, isolated=0.05, hub_deg=N - 1)
    # unsorted rows are legal CSR too: shuffle inside a few rows
    r = np.random.default_rng(seed)
    indices = indices.copy()
    for i in r.choice(N, 10, replace=False):
        r.shuffle(indices[indptr[i]:indptr[i + 1]])
    got = oracle.plan(indptr, indices, T, C)
    ref = _plan_recount(indptr, indices, T, C)
    for k, v in ref.items():
        np.testing.assert_array_equal(got[k], v, err_msg=k)


def test_plan_on_powerlaw_workload():
    w = synth.WORKLOADS["powerlaw170k"]
    indptr, indices = synth.make_graph(w)
    got = oracle.plan(indptr, indices, 256, 256)
    ref = _plan_recount(indptr, indices, 256, 256)
    for k, v in ref.items():
        np.testing.assert_array_equal(got[k], v, err_msg=k)


# ----------------------------------------------------------------------------
# row-subset evaluation (used for sampled checks at full size)
# ----------------------------------------------------------------------------
def test_row_subset_matches_full():
    N, H, D = 80, 2, 4
    indptr, indices = _graph(14, N, 6.0, isolated=0.1)
    Q, K, V, G = _feats(14, N, H, D)
    out, lse = oracle.forward(indptr, indices, Q, K, V)
    dQ, dK, dV, _ = oracle.backward(indptr, indices, Q, K, V, G)
    rows = np.array([3, 17, 41, 0, 79])
    rp, col, ids = oracle.rows_subgraph(indptr, indices, rows)
    o, l = oracle.forward(rp, col, Q, K, V, rows=ids)
    np.testing.assert_array_equal(o, out[rows])
    np.testing.assert_array_equal(l, lse[rows])
    src = np.array([5, 6, 60])
    closure = oracle.sources_closure(indptr, indices, src)
    rp, col, ids = oracle.rows_subgraph(indptr, indices, closure)
    sq, sk, sv, _ = oracle.backward(rp, col, Q, K, V, G[closure], rows=ids)
    np.testing.assert_allclose(sq, dQ[closure], atol=1e-13)
    np.testing.assert_allclose(sk[src], dK[src], atol=1e-13)
    np.testing.assert_allclose(sv[src], dV[src], atol=1e-13)
