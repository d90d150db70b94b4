"""Pins of the oracle's weighted SpMM: scipy's sparse product (duplicates
summed), a hand-worked example, linearity, empty rows."""
import numpy as np
import pytest
import scipy.sparse as sp

import oracle
from gnn_sparse_attention_gb300 import synth


def test_spmm_hand_example():
    # row 0 <- 1 (w 2), 2 (w -1); row 1 <- none; row 2 <- 0 (w 0.5), 0 (w 0.5)
    ip = np.array([0, 2, 2, 4], np.int32)
    ix = np.array([1, 2, 0, 0], np.int32)
    w = np.array([2.0, -1.0, 0.5, 0.5])
    X = np.array([[1.0, 10.0], [2.0, 20.0], [3.0, 30.0]])
    y = oracle.spmm(ip, ix, w, X)
    assert y.tolist() == [[1.0, 10.0], [0.0, 0.0], [1.0, 10.0]]


@pytest.mark.parametrize("seed,N,avg,F", [(0, 300, 6.0, 16), (1, 100, 30.0, 3)])
def test_spmm_equals_scipy(seed, N, avg, F):
    ip, ix = synth.small_graph(seed, N, avg, isolated=0.1)
    ix = np.concatenate([ix, ix[:20]]).astype(np.int32)
    ip = ip.copy()
    ip[-1] += 20                                  # last row gains 20 repeated sources
    r = np.random.default_rng(seed)
    w = r.standard_normal(len(ix))
    X = r.standard_normal((N, F))
    A = sp.csr_matrix((w, ix, ip), shape=(N, N))  # csr_matrix sums repeated entries
    np.testing.assert_allclose(oracle.spmm(ip, ix, w, X), A @ X, rtol=1e-12, atol=1e-12)


def test_spmm_linearity():
    ip, ix = synth.small_graph(2, 200, 5.0)
    r = np.random.default_rng(2)
    w1, w2 = r.standard_normal(len(ix)), r.standard_normal(len(ix))
    X = r.standard_normal((200, 4))
    np.testing.assert_allclose(oracle.spmm(ip, ix, 2 * w1 + w2, X),
                               2 * oracle.spmm(ip, ix, w1, X) + oracle.spmm(ip, ix, w2, X),
                               rtol=1e-12, atol=1e-12)
