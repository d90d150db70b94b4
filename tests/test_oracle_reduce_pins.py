"""Pins of the oracle's max / min pooling (reduction-based layers) and its
backward: a numpy brute force per row, constructed ties, empty rows, the
min/max symmetry, and central finite differences (pooling is piecewise
linear, so away from ties the difference quotient is exact)."""
import numpy as np
import pytest

import oracle
from gnn_sparse_attention_gb300 import synth


def _brute(ip, ix, X, op):
    N = len(ip) - 1
    F = X.shape[1]
    out = np.zeros((N, F))
    arg = np.full((N, F), -1, np.int32)
    for i in range(N):
        js = ix[ip[i]:ip[i + 1]]
        if len(js) == 0:
            continue
        vals = X[js]                                   # [deg, F]
        best = vals.max(axis=0) if op == oracle.MAX else vals.min(axis=0)
        out[i] = best
        for f in range(F):
            arg[i, f] = min(int(j) for j, v in zip(js, vals[:, f]) if v == best[f])
    return out, arg


@pytest.mark.parametrize("op", [oracle.MAX, oracle.MIN])
@pytest.mark.parametrize("seed,N,avg,F", [(0, 50, 4.0, 8), (1, 200, 12.0, 3), (2, 80, 1.0, 16)])
def test_pooling_brute_force(op, seed, N, avg, F):
    ip, ix = synth.small_graph(seed, N, avg, isolated=0.1)
    X = np.random.default_rng(seed).standard_normal((N, F))
    out, arg = oracle.reduce_forward(ip, ix, X, op)
    bo, ba = _brute(ip, ix, X, op)
    np.testing.assert_array_equal(out, bo)
    np.testing.assert_array_equal(arg, ba)


def test_pooling_ties_pick_the_smallest_source():
    # row 0 <- sources 5, 2, 9, 2 (a repeated edge); all features tie at 1.0
    ip = np.array([0, 4, 4], np.int32)
    ix = np.array([5, 2, 9, 2], np.int32)
    X = np.zeros((10, 3))
    X[[5, 2, 9]] = 1.0
    X[9, 2] = 3.0
    out, arg = oracle.reduce_forward(ip, ix, X, oracle.MAX)
    assert out[0].tolist() == [1.0, 1.0, 3.0]
    assert arg[0].tolist() == [2, 2, 9]
    assert out[1].tolist() == [0.0, 0.0, 0.0] and arg[1].tolist() == [-1, -1, -1]
    out, arg = oracle.reduce_forward(ip, ix, X, oracle.MIN)
    assert out[0].tolist() == [1.0, 1.0, 1.0] and arg[0].tolist() == [2, 2, 2]


def test_min_is_negated_max_of_negation():
    ip, ix = synth.small_graph(3, 120, 6.0, isolated=0.05)
    X = np.random.default_rng(3).standard_normal((120, 5))
    mo, ma = oracle.reduce_forward(ip, ix, -X, oracle.MAX)
    no, na = oracle.reduce_forward(ip, ix, X, oracle.MIN)
    np.testing.assert_array_equal(no, -mo + 0.0)
    np.testing.assert_array_equal(na, ma)


@pytest.mark.parametrize("op", [oracle.MAX, oracle.MIN])
def test_pooling_backward_finite_differences(op):
    ip, ix = synth.small_graph(4, 40, 5.0, isolated=0.1)
    N, F = 40, 4
    r = np.random.default_rng(4)
    X = r.standard_normal((N, F))
    G = r.standard_normal((N, F))
    _, arg = oracle.reduce_forward(ip, ix, X, op)
    dx = oracle.reduce_backward(arg, G, N)
    h = 1e-7
    for j in range(N):
        for f in range(F):
            Xp, Xm = X.copy(), X.copy()
            Xp[j, f] += h
            Xm[j, f] -= h
            lp = (oracle.reduce_forward(ip, ix, Xp, op)[0] * G).sum()
            lm = (oracle.reduce_forward(ip, ix, Xm, op)[0] * G).sum()
            assert abs((lp - lm) / (2 * h) - dx[j, f]) < 1e-6
