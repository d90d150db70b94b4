"""Seeded synthetic graphs and feature tensors.

This module holds no attention arithmetic: it only draws graphs and
features.  It is the one piece that both the CUDA path's tests/benchmark and
the fp64 oracle consume.

The evaluation graphs of "On Efficient Scaling of GNNs via IO-Aware Layers
Implementations" (OGB, citation networks, GraphLand industrial graphs; zh/ko
technical summaries, "Experimental results") are not available here; the
generators below stand in for them with matching node count, edge count and
degree shape.  Every graph is CSR by destination: row i lists the sources j
of the edges j -> i in ascending order.

Every draw comes from its own numpy sub-stream ``SeedSequence([seed, s])``:
s = 0 graph, 1 Q (or xl), 2 K (or xr), 3 V, 4 dO, 5 a.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

STREAM_GRAPH, STREAM_Q, STREAM_K, STREAM_V, STREAM_DO, STREAM_A = range(6)


def rng_for(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: graph recipe + head layout + I/O dtype."""
    name: str
    graph: str               # "er" | "zipf" | "lognormal" | "sbm"
    N: int
    H: int
    D: int
    dtype: str               # "f32" | "bf16"
    score: str               # "dot" | "gatv2"
    self_loops: bool = False
    params: dict = field(default_factory=dict)


WORKLOADS = {
    # Erdos-Renyi directed, avg in-degree 8 plus self-loops; correctness case.
    "er1k": Workload("er1k", "er", 1024, 2, 16, "f32", "dot", True, {"avg": 8.0}),
    # Power-law in-degrees Zipf(2.1) capped at 13000, 1.2M edges plus self-loops.
    "powerlaw170k": Workload("powerlaw170k", "zipf", 170_000, 8, 16, "bf16", "dot", True,
                             {"alpha": 2.1, "cap": 13_000, "edges": 1_200_000}),
    # Lognormal in-degrees (mu 5.5, sigma 1.2), avg ~500, hubs of 1e4..5e4.
    "lognormal233k": Workload("lognormal233k", "lognormal", 233_000, 4, 32, "bf16", "dot",
                              False, {"mu": 5.5, "sigma": 1.2}),
    # GATv2 on a Zipf(2.3) power-law graph with 62M edges.
    "gatv2_powerlaw2m4": Workload("gatv2_powerlaw2m4", "zipf", 2_400_000, 4, 32, "bf16",
                                  "gatv2", False,
                                  {"alpha": 2.3, "cap": 2_399_999, "edges": 62_000_000}),
    # The same GATv2 recipe on a quarter of the nodes and edges (profiling-sized case).
    "gatv2_powerlaw600k": Workload("gatv2_powerlaw600k", "zipf", 600_000, 4, 32, "bf16",
                                   "gatv2", False,
                                   {"alpha": 2.3, "cap": 599_999, "edges": 15_500_000}),
    # Stochastic block model, 64-node communities ordered by community.
    "sbm1m": Workload("sbm1m", "sbm", 1 << 20, 8, 64, "bf16", "dot", False,
                      {"block": 64, "p_in": 0.5, "inter_per_node": 4}),
    # The same block model on a quarter of the nodes (profiling-sized case).
    "sbm256k": Workload("sbm256k", "sbm", 1 << 18, 8, 64, "bf16", "dot", False,
                        {"block": 64, "p_in": 0.5, "inter_per_node": 4}),
}


# ----------------------------------------------------------------------------
# degree sequences
# ----------------------------------------------------------------------------
def zipf_degrees(rng, n, alpha, lo, hi):
    """n draws of a Zipf law P(k) ~ k^-alpha truncated to [lo, hi]."""
    k = np.arange(lo, hi + 1, dtype=np.float64)
    cdf = np.cumsum(k ** -alpha)
    cdf /= cdf[-1]
    u = rng.random(n)
    return (lo + np.searchsorted(cdf, u, side="left")).astype(np.int64)


def rescale_degrees(d, total, cap):
    """Scale a degree sequence so it sums to ``total`` exactly, capped at ``cap``.

    Proportional scaling, floors, then the remaining units go to the largest
    fractional parts (largest-remainder rounding, ties by index).  Nodes that
    would exceed ``cap`` are pinned at ``cap`` and the rest re-scaled.
    """
    d = np.asarray(d, np.float64)
    pinned = np.zeros(len(d), bool)
    while True:
        free_total = total - cap * int(pinned.sum())
        x = np.where(pinned, float(cap), d * (free_total / d[~pinned].sum()))
        over = (~pinned) & (x > cap)
        if over.any():
            pinned |= over
            continue
        out = np.floor(x).astype(np.int64)
        out[pinned] = cap
        rem = total - int(out.sum())
        frac = np.where(pinned, -1.0, x - np.floor(x))
        order = np.argsort(-frac, kind="stable")
        out[order[:rem]] += 1
        if out.max() > cap:  # a +1 pushed a node over the cap: pin and redo
            pinned |= out > cap
            continue
        return out


# ----------------------------------------------------------------------------
# edge sampling
# ----------------------------------------------------------------------------
def _sorted_unique_sources(rng, N, deg):
    """For each row i, deg[i] distinct sources j != i drawn uniformly, sorted.

    Returns (indptr int64 [N+1], indices int32 [M]).
    """
    deg = np.asarray(deg, np.int64)
    if (deg > N - 1).any():
        raise ValueError("degree exceeds N-1")
    indptr = np.zeros(N + 1, np.int64)
    np.cumsum(deg, out=indptr[1:])
    M = int(indptr[-1])
    indices = np.empty(M, np.int64)
    dense = deg > (N - 1) // 8
    # dense rows: exact sampling without replacement, row by row
    for i in np.nonzero(dense)[0]:
        c = rng.choice(N - 1, size=int(deg[i]), replace=False)
        c = c + (c >= i)
        indices[indptr[i]:indptr[i + 1]] = np.sort(c)
    # sparse rows: draw with replacement, then redraw duplicates until none
    rows = np.nonzero(~dense)[0]
    if len(rows) and deg[rows].sum() > 0:
        dsub = deg[rows]
        dst = np.repeat(rows, dsub)
        src = rng.integers(0, N - 1, size=len(dst), dtype=np.int64)
        src += src >= dst
        key = np.sort(dst * N + src)
        del dst, src
        seg_start = np.cumsum(dsub) - dsub          # row segments inside ``key``
        while True:
            dup = np.nonzero(key[1:] == key[:-1])[0] + 1
            if len(dup) == 0:
                break
            d_dst = key[dup] // N
            new = rng.integers(0, N - 1, size=len(dup), dtype=np.int64)
            new += new >= d_dst
            key[dup] = d_dst * N + new
            # keys are destination-major, so re-sorting the affected rows'
            # segments together puts every row back into its own segment
            r = np.searchsorted(rows, np.unique(d_dst))
            pos = np.repeat(seg_start[r], dsub[r]) + (
                np.arange(int(dsub[r].sum())) - np.repeat(np.cumsum(dsub[r]) - dsub[r], dsub[r]))
            key[pos] = np.sort(key[pos])
        pos = np.repeat(indptr[rows], dsub) + (np.arange(len(key)) - np.repeat(seg_start, dsub))
        indices[pos] = key % N
    return indptr, indices


def _add_self_loops(indptr, indices):
    N = len(indptr) - 1
    deg = np.diff(indptr)
    dst = np.repeat(np.arange(N, dtype=np.int64), deg)
    key = np.concatenate([dst * N + indices, np.arange(N, dtype=np.int64) * (N + 1)])
    key.sort()
    new_ptr = np.zeros(N + 1, np.int64)
    np.cumsum(deg + 1, out=new_ptr[1:])
    return new_ptr, key % N


def make_graph(w: Workload, seed: int = 0):
    """(indptr int32 [N+1], indices int32 [M]) for a workload."""
    rng = rng_for(seed, STREAM_GRAPH)
    N, p = w.N, w.params
    if w.graph == "er":
        prob = p["avg"] / (N - 1)
        mask = rng.random((N, N)) < prob          # mask[i, j]: edge j -> i
        np.fill_diagonal(mask, False)
        deg = mask.sum(axis=1)
        indptr = np.zeros(N + 1, np.int64)
        np.cumsum(deg, out=indptr[1:])
        indices = np.nonzero(mask)[1].astype(np.int64)
    elif w.graph == "zipf":
        d = zipf_degrees(rng, N, p["alpha"], 1, p["cap"])
        d = rescale_degrees(d, p["edges"], p["cap"])
        indptr, indices = _sorted_unique_sources(rng, N, d)
    elif w.graph == "lognormal":
        d = np.clip(np.rint(np.exp(rng.normal(p["mu"], p["sigma"], N))), 0, N - 1)
        indptr, indices = _sorted_unique_sources(rng, N, d.astype(np.int64))
    elif w.graph == "sbm":
        B = p["block"]
        nb = N // B
        keys = []
        # intra-community: ordered pairs (j -> i), i != j, kept with p_in
        for b0 in range(0, nb, 4096):
            b1 = min(nb, b0 + 4096)
            m = rng.random((b1 - b0, B, B)) < p["p_in"]     # m[b, i, j]: j -> i
            m[:, np.arange(B), np.arange(B)] = False
            bb, ii, jj = np.nonzero(m)
            base = (bb + b0).astype(np.int64) * B
            keys.append((base + ii) * N + (base + jj))
        # inter-community: uniform destination, uniform source outside it
        n_inter = p["inter_per_node"] * N
        dst = rng.integers(0, N, size=n_inter, dtype=np.int64)
        other = rng.integers(0, N - B, size=n_inter, dtype=np.int64)
        start = (dst // B) * B
        src = other + (other >= start) * B
        keys.append(dst * N + src)
        key = np.unique(np.concatenate(keys))
        dst_all = key // N
        indptr = np.zeros(N + 1, np.int64)
        np.cumsum(np.bincount(dst_all, minlength=N), out=indptr[1:])
        indices = key % N
    else:
        raise ValueError(w.graph)
    if w.self_loops:
        indptr, indices = _add_self_loops(indptr, indices)
    if indptr[-1] >= 2 ** 31:
        raise ValueError("graph too large for int32 edge ids")
    return indptr.astype(np.int32), indices.astype(np.int32)


# ----------------------------------------------------------------------------
# features
# ----------------------------------------------------------------------------
def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """fp32 N(0, std^2) draws of the given shape from sub-stream ``stream``."""
    x = rng_for(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def make_features(w: Workload, seed: int = 0, N: int | None = None):
    """Dict of fp32 numpy arrays: Q, K, V, dO [N, H, D] and a [H, D] (GATv2)."""
    N = w.N if N is None else N
    shape = (N, w.H, w.D)
    f = {
        "Q": normal(seed, STREAM_Q, shape),
        "K": normal(seed, STREAM_K, shape),
        "V": normal(seed, STREAM_V, shape),
        "dO": normal(seed, STREAM_DO, shape),
    }
    if w.score == "gatv2":
        f["a"] = normal(seed, STREAM_A, (w.H, w.D), std=float(1.0 / np.sqrt(w.D)))
    return f


def small_graph(seed: int, N: int, avg: float, isolated: float = 0.0, hub_deg: int = 0,
                self_loops: bool = False):
    """Small random graph for parity tests: ER-like rows, optional isolated
    nodes (fraction) and one hub row (node 0) of ``hub_deg`` sources."""
    rng = rng_for(seed, STREAM_GRAPH)
    deg = rng.poisson(avg, N).astype(np.int64)
    deg = np.minimum(deg, N - 1)
    if isolated > 0:
        deg[rng.random(N) < isolated] = 0
    if hub_deg:
        deg[0] = min(hub_deg, N - 1)
    indptr, indices = _sorted_unique_sources(rng, N, deg)
    if self_loops:
        indptr, indices = _add_self_loops(indptr, indices)
    return indptr.astype(np.int32), indices.astype(np.int32)
