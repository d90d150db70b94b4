"""Pins of the oracle's dense-tile split (the tensor-core path's plan).

Each check recounts the split from its definition with plain Python
dictionaries over the edge list: blocks of 128 x 128 node ids, a block with at
least min_count edges is a tile, pairs seen once in a tile are its mask bits,
everything else is the residual CSR in CSR order.
"""
from collections import Counter

import numpy as np
import pytest

import oracle


def _csr(N, edges):
    """CSR of (dst, src) pairs, rows in the given order of appearance."""
    rows = [[] for _ in range(N)]
    for i, j in edges:
        rows[i].append(j)
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    return indptr, indices


def _recount(indptr, indices, min_count):
    N = len(indptr) - 1
    edges = [(i, int(indices[e])) for i in range(N) for e in range(indptr[i], indptr[i + 1])]
    block = Counter((i // 128, j // 128) for i, j in edges)
    tiles = sorted(b for b, n in block.items() if n >= min_count)
    pairs = Counter(edges)
    masks = {}
    for t in tiles:
        m = np.zeros((128, 4), np.uint32)
        for (i, j), n in pairs.items():
            if (i // 128, j // 128) == t and n == 1:
                m[i % 128, (j % 128) // 32] |= np.uint32(1 << (j % 32))
        masks[t] = m
    tile_set = set(tiles)
    res_rows = [[j for (ii, j) in edges if ii == i
                 and not ((i // 128, j // 128) in tile_set and pairs[(i, j)] == 1)]
                for i in range(N)]
    return tiles, masks, res_rows


def _check(indptr, indices, min_count):
    got = oracle.tile_plan(indptr, indices, min_count)
    tiles, masks, res_rows = _recount(indptr, indices, min_count)
    assert list(zip(got["tile_rb"].tolist(), got["tile_cb"].tolist())) == tiles
    for k, t in enumerate(tiles):
        np.testing.assert_array_equal(got["masks"][k], masks[t])
    want_ptr = np.concatenate([[0], np.cumsum([len(r) for r in res_rows])])
    np.testing.assert_array_equal(got["indptr_r"], want_ptr)
    np.testing.assert_array_equal(got["indices_r"], [j for r in res_rows for j in r])
    return got


def _random_graph(seed, N, dense_blocks, p_dense, n_sparse, n_dup):
    r = np.random.default_rng(seed)
    edges = []
    for rb, cb in dense_blocks:
        for i in range(rb * 128, min(N, rb * 128 + 128)):
            for j in range(cb * 128, min(N, cb * 128 + 128)):
                if r.random() < p_dense:
                    edges.append((i, j))
    for _ in range(n_sparse):
        edges.append((int(r.integers(N)), int(r.integers(N))))
    for _ in range(n_dup):  # repeat some existing pairs (multi-edges)
        edges.append(edges[int(r.integers(len(edges)))])
    order = r.permutation(len(edges))
    return _csr(N, [edges[k] for k in order])


@pytest.mark.parametrize("seed,N,blocks,p,sparse,dup,mc", [
    (0, 300, [(0, 0), (1, 2), (2, 1)], 0.3, 400, 30, 1000),
    (1, 256, [(0, 1), (1, 1)], 0.05, 200, 10, 700),
    (2, 200, [(0, 0)], 0.5, 50, 40, 1),
    (3, 390, [(0, 0), (1, 1), (2, 2), (3, 0)], 0.2, 1000, 0, 16384),
])
def test_tile_split_recount(seed, N, blocks, p, sparse, dup, mc):
    _check(*_random_graph(seed, N, blocks, p, sparse, dup), mc)


def test_tile_threshold_is_inclusive():
    edges = [(i, j) for i in range(10) for j in range(10)]      # 100 edges in block (0, 0)
    ip, ix = _csr(140, edges + [(130, 3)])
    assert len(oracle.tile_plan(ip, ix, 100)["tile_rb"]) == 1
    assert len(oracle.tile_plan(ip, ix, 101)["tile_rb"]) == 0


def test_tile_duplicates_stay_residual():
    edges = [(i, j) for i in range(8) for j in range(8)] + [(3, 5), (3, 5), (7, 0)]
    ip, ix = _csr(8, edges)
    got = _check(ip, ix, 10)
    m = got["masks"][0]
    assert not (m[3, 0] >> 5) & 1 and not m[7, 0] & 1     # repeated pairs: no bit
    assert got["indices_r"].tolist() == [5, 5, 5, 0, 0]   # all copies, in CSR order
    assert int(m.view(np.uint8).sum()) > 0


def test_tile_edges_and_residual_partition_the_edges():
    ip, ix = _random_graph(5, 260, [(0, 0), (1, 0), (2, 2)], 0.25, 300, 20)
    got = oracle.tile_plan(ip, ix, 500)
    tile_edges = Counter()
    for rb, cb, m in zip(got["tile_rb"], got["tile_cb"], got["masks"]):
        for r in range(128):
            for c in range(128):
                if (int(m[r, c // 32]) >> (c % 32)) & 1:
                    tile_edges[(int(rb) * 128 + r, int(cb) * 128 + c)] += 1
    res = Counter((i, int(got["indices_r"][e])) for i in range(len(ip) - 1)
                  for e in range(got["indptr_r"][i], got["indptr_r"][i + 1]))
    orig = Counter((i, int(ix[e])) for i in range(len(ip) - 1) for e in range(ip[i], ip[i + 1]))
    assert tile_edges + res == orig
    assert len(tile_edges) > 0


def test_tile_min_count_rounding():
    assert oracle.tile_min_count(0.0625) == 1024
    assert oracle.tile_min_count(1.0) == 16384
    assert oracle.tile_min_count(1e-9) == 1
    assert oracle.tile_min_count(0.1) == 1639      # 0.1f = 0.100000001490116...
