"""Pins of the oracle's node relabelling (degree order, reverse Cuthill-McKee)
and of the relabelled graph.

The RCM checks do not rerun the algorithm: they verify that the unreversed
order is a breadth-first order with the stated root and tie rules (every
component starts at the least-(degree, id) node left, nodes appear in
non-decreasing order of their BFS parent's position, siblings by (degree,
id)), plus textbook cases and the bandwidth a relabelling is meant to cut.
"""
import numpy as np
import pytest
import scipy.sparse as sp

import oracle
from gnn_sparse_attention_gb300 import synth


def _csr(N, edges):
    rows = [[] for _ in range(N)]
    for i, j in edges:
        rows[i].append(j)
    ptr = np.zeros(N + 1, np.int32)
    ptr[1:] = np.cumsum([len(r) for r in rows])
    return ptr, np.array([j for r in rows for j in r], np.int32)


def _undirected(ip, ix):
    N = len(ip) - 1
    adj = [set() for _ in range(N)]
    for i in range(N):
        for j in ix[ip[i]:ip[i + 1]]:
            if j != i:
                adj[i].add(int(j))
                adj[int(j)].add(i)
    return adj


def _check_cm(ip, ix, perm):
    N = len(ip) - 1
    assert sorted(perm.tolist()) == list(range(N))
    adj = _undirected(ip, ix)
    deg = [len(a) for a in adj]
    order = perm[::-1].tolist()                 # Cuthill-McKee order
    pos = {v: k for k, v in enumerate(order)}
    parent = {}
    for k, v in enumerate(order):
        earlier = [pos[w] for w in adj[v] if pos[w] < k]
        if not earlier:                          # a component root
            rest = order[k:]
            assert (deg[v], v) == min((deg[u], u) for u in rest)
            parent[v] = None
        else:
            parent[v] = min(earlier)
    for k in range(1, N):
        u, v = order[k - 1], order[k]
        if parent[u] is None or parent[v] is None:
            continue
        assert parent[u] <= parent[v]
        if parent[u] == parent[v]:
            assert (deg[u], u) < (deg[v], v)


def _bandwidth(ip, ix, perm):
    inv = np.empty(len(perm), np.int64)
    inv[perm] = np.arange(len(perm))
    b = 0
    for i in range(len(ip) - 1):
        for j in ix[ip[i]:ip[i + 1]]:
            b = max(b, abs(int(inv[i]) - int(inv[j])))
    return b


def test_rcm_path_and_star():
    ip, ix = _csr(5, [(1, 0), (2, 1), (3, 2), (4, 3)])
    assert oracle.reorder(ip, ix, oracle.REORDER_RCM).tolist() == [4, 3, 2, 1, 0]
    # star around node 2: root = leaf 0 (degree 1), then the centre, then the
    # other leaves by id; reversed
    ip, ix = _csr(5, [(2, 0), (2, 1), (3, 2), (4, 2)])
    assert oracle.reorder(ip, ix, oracle.REORDER_RCM).tolist() == [4, 3, 1, 2, 0]


@pytest.mark.parametrize("seed,N,avg", [(0, 60, 3.0), (1, 200, 1.2), (2, 150, 8.0)])
def test_rcm_is_a_cuthill_mckee_order(seed, N, avg):
    ip, ix = synth.small_graph(seed, N, avg, isolated=0.1)
    _check_cm(ip, ix, oracle.reorder(ip, ix, oracle.REORDER_RCM))


def test_rcm_cuts_the_bandwidth_of_a_shuffled_grid():
    k = 12
    r = np.random.default_rng(3)
    lab = r.permutation(k * k)
    edges = []
    for a in range(k):
        for b in range(k):
            if a + 1 < k:
                edges.append((lab[a * k + b], lab[(a + 1) * k + b]))
            if b + 1 < k:
                edges.append((lab[a * k + b], lab[a * k + b + 1]))
    ip, ix = _csr(k * k, edges)
    perm = oracle.reorder(ip, ix, oracle.REORDER_RCM)
    _check_cm(ip, ix, perm)
    assert _bandwidth(ip, ix, perm) <= k + 1
    assert _bandwidth(ip, ix, np.arange(k * k)) > 4 * k
    # scipy's RCM (another start rule) reaches the same order of bandwidth
    a = sp.csr_matrix((np.ones(len(ix)), ix, ip), shape=(k * k, k * k))
    sym = ((a + a.T) > 0).astype(np.int8).tocsr()
    from scipy.sparse.csgraph import reverse_cuthill_mckee
    ref = reverse_cuthill_mckee(sym, symmetric_mode=True)
    assert _bandwidth(ip, ix, perm) <= _bandwidth(ip, ix, np.asarray(ref, np.int32)) + 1


def test_degree_order():
    ip, ix = synth.small_graph(4, 300, 5.0, hub_deg=120)
    perm = oracle.reorder(ip, ix, oracle.REORDER_DEGREE)
    N = len(ip) - 1
    assert sorted(perm.tolist()) == list(range(N))
    tot = np.diff(ip).astype(np.int64) + np.bincount(ix, minlength=N)
    keys = [(-int(tot[v]), int(v)) for v in perm]
    assert keys == sorted(keys)
    assert perm[0] == int(np.argmax(tot))


def test_permuted_csr_is_the_relabelled_graph():
    ip, ix = synth.small_graph(5, 120, 4.0, isolated=0.05)
    N = len(ip) - 1
    rows = [list(ix[ip[i]:ip[i + 1]]) for i in range(N)]
    rows[7] += rows[7][:2] + [3, 3]                      # repeated sources
    ip, ix = _csr(N, [(i, j) for i in range(N) for j in rows[i]])
    r = np.random.default_rng(0)
    perm = r.permutation(N).astype(np.int32)
    ptr, idx = oracle.permute_csr(ip, ix, perm)
    inv = np.empty(N, np.int64)
    inv[perm] = np.arange(N)
    for i in range(N):
        old = perm[i]
        want = sorted(int(inv[j]) for j in ix[ip[old]:ip[old + 1]])
        assert idx[ptr[i]:ptr[i + 1]].tolist() == want


@pytest.mark.parametrize("method", [oracle.REORDER_DEGREE, oracle.REORDER_RCM])
def test_attention_is_equivariant_under_relabelling(method):
    ip, ix = synth.small_graph(6, 80, 5.0, isolated=0.1)
    N = len(ip) - 1
    w = synth.Workload("t", "er", N, 2, 8, "f32", "dot")
    f = synth.make_features(w, seed=2)
    Q, K, V = (f[k].astype(np.float64) for k in ("Q", "K", "V"))
    out, lse = oracle.forward(ip, ix, Q, K, V)
    perm = oracle.reorder(ip, ix, method)
    ptr, idx = oracle.permute_csr(ip, ix, perm)
    out_p, lse_p = oracle.forward(ptr, idx, Q[perm], K[perm], V[perm])
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse_p), np.isneginf(lse[perm]))
    fin = np.isfinite(lse_p)
    np.testing.assert_allclose(lse_p[fin], lse[perm][fin], rtol=1e-12)
