/*
 * gattn_oracle.c -- plain fp64 CPU oracle for fused CSR graph attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or constant with
 * the CUDA library; the two meet only in the seeded input generators.
 *
 * What it computes (source: "On Efficient Scaling of GNNs via IO-Aware
 * Layers Implementations", zh and ko technical summaries, section
 * "Methodology", attention-based layers):
 *   the attention layer scores every in-neighbour j of a destination i,
 *   normalises the scores with a softmax over the neighbourhood and sums the
 *   neighbours' values with those weights.  The fused method streams this
 *   with an online softmax and keeps a per-node log-sum-exp for the backward;
 *   its result equals the plain definition below up to rounding order, so
 *   the oracle is that definition written out: it MATERIALISES the O(M*H)
 *   edge logits and probabilities that the fused kernels avoid.
 *
 * Score functions (the two layer types the pages name, Graph Transformer
 * and GATv2; formulas as fixed by the build contract because the pages
 * print none):
 *   dot   : s_ijh = scale * sum_d q_ihd k_jhd            (scale = 1/sqrt(D))
 *   GATv2 : s_ijh = sum_d a_hd * LeakyReLU(q_ihd + k_jhd) (q = xl, k = xr)
 * with LeakyReLU(z) = z for z > 0, slope*z otherwise, and its derivative
 * 1 for z > 0, slope otherwise.
 *
 * Readings where the pages are silent (listed in the design notes too):
 *   - a node with no in-edges gets out = 0 and lse = -inf;
 *   - i is the destination (row of the CSR), j the source (column);
 *   - no bias, no head concat/mean: outputs are per head [rows, H, D].
 *
 * Layouts: every dense tensor is row-major [nodes, H, D] fp64.  The graph is
 * given as a list of destination rows: row r is node row_ids[r] (or r when
 * row_ids is NULL), its in-edges are col[row_ptr[r] .. row_ptr[r+1]).  A
 * subset of rows is allowed: forward rows are independent, so the oracle
 * on a subset of rows gives the exact values of those rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_DOT 0
#define ORC_GATV2 1

static double leaky(double z, double slope) { return z > 0.0 ? z : slope * z; }
static double leaky_grad(double z, double slope) { return z > 0.0 ? 1.0 : slope; }

/* One edge, one head: the score s_ijh. q and k point at the head's D values. */
static double edge_score(int kind, int D, double scale, const double* a_h, double slope,
                         const double* q, const double* k) {
  double s = 0.0;
  if (kind == ORC_DOT) {
    for (int d = 0; d < D; ++d) s += q[d] * k[d];
    return scale * s;
  }
  for (int d = 0; d < D; ++d) s += a_h[d] * leaky(q[d] + k[d], slope);
  return s;
}

static int64_t node_of(const int32_t* row_ids, int64_t r) { return row_ids ? (int64_t)row_ids[r] : r; }

/*
 * Materialise the edge logits e[nnz, H] and the softmax probabilities
 * p[nnz, H]; write lse[n_rows, H].  Returns 0, or -1 on allocation failure.
 */
static int logits_and_probs(int64_t n_rows, const int32_t* row_ids, const int64_t* row_ptr,
                            const int32_t* col, int H, int D, int kind, double scale,
                            const double* a, double slope, const double* Q, const double* K,
                            double* p, double* lse) {
  const int64_t HD = (int64_t)H * D;
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t i = node_of(row_ids, r);
    const int64_t e0 = row_ptr[r], e1 = row_ptr[r + 1];
    for (int h = 0; h < H; ++h) {
      const double* q = Q + i * HD + (int64_t)h * D;
      const double* a_h = a ? a + (int64_t)h * D : NULL;
      /* logits */
      for (int64_t e = e0; e < e1; ++e) {
        const double* k = K + (int64_t)col[e] * HD + (int64_t)h * D;
        p[e * H + h] = edge_score(kind, D, scale, a_h, slope, q, k);
      }
      if (e1 == e0) { /* isolated destination: reading, lse = -inf */
        lse[r * H + h] = -INFINITY;
        continue;
      }
      /* softmax over the neighbourhood */
      double m = -INFINITY;
      for (int64_t e = e0; e < e1; ++e) m = fmax(m, p[e * H + h]);
      double z = 0.0;
      for (int64_t e = e0; e < e1; ++e) z += exp(p[e * H + h] - m);
      for (int64_t e = e0; e < e1; ++e) p[e * H + h] = exp(p[e * H + h] - m) / z;
      lse[r * H + h] = m + log(z);
    }
  }
  return 0;
}

/*
 * Forward: out[r] = sum_j p_ij v_j per head, lse[r] = log sum_j exp(s_ij).
 * out is [n_rows, H, D] indexed by row position r; lse is [n_rows, H].
 */
int oracle_forward(int64_t n_rows, const int32_t* row_ids, const int64_t* row_ptr,
                   const int32_t* col, int H, int D, int kind, double scale, const double* a,
                   double slope, const double* Q, const double* K, const double* V, double* out,
                   double* lse) {
  const int64_t HD = (int64_t)H * D;
  const int64_t nnz = row_ptr[n_rows];
  double* p = (double*)malloc((size_t)(nnz > 0 ? nnz : 1) * (size_t)H * sizeof(double));
  if (!p) return -1;
  logits_and_probs(n_rows, row_ids, row_ptr, col, H, D, kind, scale, a, slope, Q, K, p, lse);
  for (int64_t r = 0; r < n_rows; ++r) {
    double* o = out + r * HD;
    memset(o, 0, (size_t)HD * sizeof(double));
    for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
      const double* v = V + (int64_t)col[e] * HD;
      for (int h = 0; h < H; ++h) {
        const double w = p[e * H + h];
        for (int d = 0; d < D; ++d) o[h * D + d] += w * v[h * D + d];
      }
    }
  }
  free(p);
  return 0;
}

/*
 * Analytic backward of L = sum out * dO (dO given per row position r).
 *   dp_ij = dO_i . v_j                         (per head)
 *   ds_ij = p_ij (dp_ij - sum_k p_ik dp_ik)    (softmax Jacobian)
 *   dQ_i += ds_ij * ds/dq_i,  dK_j += ds_ij * ds/dk_j,  dV_j += p_ij dO_i,
 *   da   += ds_ij * ds/da     (GATv2 only)
 * dQ is [n_rows, H, D] by row position; dK, dV are [N, H, D] by node id and
 * are overwritten (zeroed here first); da is [H, D] (may be NULL for dot).
 * The scatter into dK/dV runs serially in edge order.
 */
int oracle_backward(int64_t n_rows, const int32_t* row_ids, const int64_t* row_ptr,
                    const int32_t* col, int64_t N, int H, int D, int kind, double scale,
                    const double* a, double slope, const double* Q, const double* K,
                    const double* V, const double* dO, double* dQ, double* dK, double* dV,
                    double* da) {
  const int64_t HD = (int64_t)H * D;
  const int64_t nnz = row_ptr[n_rows];
  const size_t eh = (size_t)(nnz > 0 ? nnz : 1) * (size_t)H;
  double* p = (double*)malloc(eh * sizeof(double));
  double* ds = (double*)malloc(eh * sizeof(double));
  double* lse = (double*)malloc((size_t)(n_rows > 0 ? n_rows : 1) * (size_t)H * sizeof(double));
  if (!p || !ds || !lse) { free(p); free(ds); free(lse); return -1; }
  logits_and_probs(n_rows, row_ids, row_ptr, col, H, D, kind, scale, a, slope, Q, K, p, lse);

  memset(dQ, 0, (size_t)n_rows * (size_t)HD * sizeof(double));
  memset(dK, 0, (size_t)N * (size_t)HD * sizeof(double));
  memset(dV, 0, (size_t)N * (size_t)HD * sizeof(double));
  if (da) memset(da, 0, (size_t)HD * sizeof(double));

  /* ds = p * (dp - sum_k p dp) */
  for (int64_t r = 0; r < n_rows; ++r) {
    const double* g = dO + r * HD;
    for (int h = 0; h < H; ++h) {
      double delta = 0.0;
      for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
        const double* v = V + (int64_t)col[e] * HD + (int64_t)h * D;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += g[h * D + d] * v[d];
        ds[e * H + h] = dp; /* dp for now */
        delta += p[e * H + h] * dp;
      }
      for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e)
        ds[e * H + h] = p[e * H + h] * (ds[e * H + h] - delta);
    }
  }

  /* chain rule through the score, edge by edge */
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t i = node_of(row_ids, r);
    const double* g = dO + r * HD;
    for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
      const int64_t j = col[e];
      for (int h = 0; h < H; ++h) {
        const double w = ds[e * H + h];
        const double pe = p[e * H + h];
        const double* q = Q + i * HD + (int64_t)h * D;
        const double* k = K + j * HD + (int64_t)h * D;
        double* dq = dQ + r * HD + (int64_t)h * D;
        double* dk = dK + j * HD + (int64_t)h * D;
        double* dv = dV + j * HD + (int64_t)h * D;
        for (int d = 0; d < D; ++d) dv[d] += pe * g[h * D + d];
        if (kind == ORC_DOT) {
          for (int d = 0; d < D; ++d) {
            dq[d] += w * scale * k[d];
            dk[d] += w * scale * q[d];
          }
        } else {
          const double* a_h = a + (int64_t)h * D;
          for (int d = 0; d < D; ++d) {
            const double z = q[d] + k[d];
            const double gz = w * a_h[d] * leaky_grad(z, slope);
            dq[d] += gz;
            dk[d] += gz;
            if (da) da[h * D + d] += w * leaky(z, slope);
          }
        }
      }
    }
  }
  free(p);
  free(ds);
  free(lse);
  return 0;
}

/*
 * Plan oracle: the per-graph metadata of the degree-aware partition
 * (source: same pages, "Methodology", reduction-based layers: nodes split
 * by a degree threshold into light and heavy sets, heavy nodes tiled over
 * edge chunks; SpMM layers: the transposed adjacency cached for backward).
 * Definition, written as straightforward loops:
 *   deg[i]      = indptr[i+1] - indptr[i]
 *   hist[b]     = #{i : bin(deg[i]) = b}, bin(0) = 0, bin(d) = 1 + floor(log2 d)
 *   light       = ascending i with deg[i] <= T
 *   chunks      = for ascending i with deg[i] > T, k = 0, 1, ...:
 *                 (i, indptr[i] + kC, min(indptr[i] + (k+1)C, indptr[i+1]))
 *   CSC         = the edges stably counting-sorted by source over CSR edge
 *                 order: indptrT[N+1], csc_dst[M] (destination), csc_eid[M]
 *                 (CSR edge id); within a column ascending edge id
 *   outdeg, hist_out, light_src, src_chunks: the same on the CSC
 * Buffers are caller-allocated: light/light_src hold N entries, chunk
 * arrays hold cap_chunks triples.  counts[0..3] receive #light, #chunks,
 * #light_src, #src_chunks.  Returns 0, -1 if a chunk array is too small,
 * -2 on allocation failure.
 */
static int bin_of(int64_t d) {
  if (d <= 0) return 0;
  int b = 1;
  while (d >= 2) { d >>= 1; ++b; }
  return b;
}

static int64_t split(int32_t n, const int64_t* ptr, int32_t T, int32_t C, int32_t* light,
                     int32_t* chunks, int64_t cap, int64_t* n_light) {
  int64_t nl = 0, nc = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t d = ptr[i + 1] - ptr[i];
    if (d <= T) { light[nl++] = i; continue; }
    for (int64_t s = ptr[i]; s < ptr[i + 1]; s += C) {
      if (nc >= cap) return -1;
      const int64_t e = s + C < ptr[i + 1] ? s + C : ptr[i + 1];
      chunks[3 * nc + 0] = i;
      chunks[3 * nc + 1] = (int32_t)s;
      chunks[3 * nc + 2] = (int32_t)e;
      ++nc;
    }
  }
  *n_light = nl;
  return nc;
}

int oracle_plan(int32_t N, int64_t M, const int32_t* indptr, const int32_t* indices, int32_t T,
                int32_t C, int32_t* deg, int32_t* hist, int32_t* light, int32_t* chunks,
                int64_t cap_chunks, int32_t* indptrT, int32_t* csc_dst, int32_t* csc_eid,
                int32_t* outdeg, int32_t* hist_out, int32_t* light_src, int32_t* src_chunks,
                int64_t cap_src_chunks, int64_t* counts) {
  int64_t* ptr = (int64_t*)malloc(((size_t)N + 1) * sizeof(int64_t));
  int64_t* ptrT = (int64_t*)malloc(((size_t)N + 1) * sizeof(int64_t));
  int64_t* fill = (int64_t*)malloc(((size_t)N + 1) * sizeof(int64_t));
  if (!ptr || !ptrT || !fill) { free(ptr); free(ptrT); free(fill); return -2; }
  for (int b = 0; b < 33; ++b) hist[b] = hist_out[b] = 0;
  for (int32_t i = 0; i <= N; ++i) ptr[i] = indptr[i];
  for (int32_t i = 0; i < N; ++i) {
    deg[i] = (int32_t)(ptr[i + 1] - ptr[i]);
    hist[bin_of(deg[i])] += 1;
  }
  /* transpose: count, prefix, stable placement in CSR edge order */
  for (int32_t j = 0; j < N; ++j) outdeg[j] = 0;
  for (int64_t e = 0; e < M; ++e) outdeg[indices[e]] += 1;
  ptrT[0] = 0;
  for (int32_t j = 0; j < N; ++j) ptrT[j + 1] = ptrT[j] + outdeg[j];
  for (int32_t j = 0; j <= N; ++j) { indptrT[j] = (int32_t)ptrT[j]; fill[j] = ptrT[j]; }
  for (int32_t i = 0; i < N; ++i)
    for (int64_t e = ptr[i]; e < ptr[i + 1]; ++e) {
      const int32_t j = indices[e];
      csc_dst[fill[j]] = i;
      csc_eid[fill[j]] = (int32_t)e;
      fill[j] += 1;
    }
  for (int32_t j = 0; j < N; ++j) hist_out[bin_of(outdeg[j])] += 1;

  int64_t nl = 0, nls = 0;
  const int64_t nc = split(N, ptr, T, C, light, chunks, cap_chunks, &nl);
  const int64_t ncs = split(N, ptrT, T, C, light_src, src_chunks, cap_src_chunks, &nls);
  free(ptr);
  free(ptrT);
  free(fill);
  if (nc < 0 || ncs < 0) return -1;
  counts[0] = nl;
  counts[1] = nc;
  counts[2] = nls;
  counts[3] = ncs;
  return 0;
}

/*
 * Dense-tile split of the CSR for the tensor-core path ("On Efficient Scaling
 * of GNNs via IO-Aware Layers Implementations", zh/ko technical summaries,
 * "Methodology", attention-based layers, tensor-core optimisation: locally
 * dense neighbourhoods are packed into block tiles so that their scores and
 * aggregation run as small dense matrix products; the remaining edges stay
 * on the CSR path).
 *
 * Reading used here: nodes are cut into blocks of 128 consecutive ids; the
 * block (rb, cb) holds the edges j -> i with i / 128 == rb and j / 128 == cb.
 * A block with at least min_count edges is a dense tile.  In a tile every
 * (i, j) pair that occurs exactly once becomes bit (j % 128) of row (i % 128)
 * of the tile's 128 x 128 mask (4 words of 32 bits per row, bit b of word w
 * is column 32 w + b); pairs that occur more than once, and every edge of a
 * block that is not a tile, form the residual CSR, kept in CSR order.  Tiles
 * are listed in (rb, cb) order.
 *
 * Outputs: tile_rb/tile_cb[n_tiles], masks[n_tiles * 512], indptr_r[N + 1],
 * indices_r[M_res].  counts[0] = n_tiles, counts[1] = M_res.  Returns 0, -1
 * if more than cap_tiles tiles, -2 on allocation failure.
 */
typedef struct { uint64_t key; int64_t e; } orc_edge_key;

static int orc_cmp_key(const void* a, const void* b) {
  const orc_edge_key* x = (const orc_edge_key*)a;
  const orc_edge_key* y = (const orc_edge_key*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return x->e < y->e ? -1 : (x->e > y->e ? 1 : 0);
}

int oracle_tile_plan(int32_t N, int64_t M, const int32_t* indptr, const int32_t* indices,
                     int64_t min_count, int64_t cap_tiles, int32_t* tile_rb, int32_t* tile_cb,
                     uint32_t* masks, int32_t* indptr_r, int32_t* indices_r, int64_t* counts) {
  const uint64_t nb = ((uint64_t)N + 127) / 128;
  orc_edge_key* ek = (orc_edge_key*)malloc((size_t)(M > 0 ? M : 1) * sizeof(orc_edge_key));
  int32_t* row = (int32_t*)malloc((size_t)(M > 0 ? M : 1) * sizeof(int32_t));
  unsigned char* in_tile = (unsigned char*)calloc((size_t)(M > 0 ? M : 1), 1);
  int32_t* pair_count = (int32_t*)malloc(128 * 128 * sizeof(int32_t));
  if (!ek || !row || !in_tile || !pair_count) {
    free(ek); free(row); free(in_tile); free(pair_count);
    return -2;
  }
  for (int32_t i = 0; i < N; ++i)
    for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) row[e] = i;
  for (int64_t e = 0; e < M; ++e) {
    ek[e].key = (uint64_t)(row[e] / 128) * nb + (uint64_t)(indices[e] / 128);
    ek[e].e = e;
  }
  qsort(ek, (size_t)M, sizeof(orc_edge_key), orc_cmp_key);

  int64_t n_tiles = 0;
  for (int64_t s = 0; s < M;) {
    int64_t t = s;
    while (t < M && ek[t].key == ek[s].key) ++t;  /* run [s, t): one block */
    if (t - s >= min_count) {
      if (n_tiles >= cap_tiles) {
        free(ek); free(row); free(in_tile); free(pair_count);
        return -1;
      }
      tile_rb[n_tiles] = (int32_t)(ek[s].key / nb);
      tile_cb[n_tiles] = (int32_t)(ek[s].key % nb);
      uint32_t* mk = masks + n_tiles * 512;
      memset(mk, 0, 512 * sizeof(uint32_t));
      memset(pair_count, 0, 128 * 128 * sizeof(int32_t));
      for (int64_t u = s; u < t; ++u) {
        const int64_t e = ek[u].e;
        pair_count[(row[e] % 128) * 128 + indices[e] % 128] += 1;
      }
      for (int64_t u = s; u < t; ++u) {
        const int64_t e = ek[u].e;
        const int r = row[e] % 128, c = indices[e] % 128;
        if (pair_count[r * 128 + c] == 1) {
          mk[r * 4 + c / 32] |= 1u << (c % 32);
          in_tile[e] = 1;
        }
      }
      ++n_tiles;
    }
    s = t;
  }
  int64_t mr = 0;
  indptr_r[0] = 0;
  for (int32_t i = 0; i < N; ++i) {
    for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e)
      if (!in_tile[e]) indices_r[mr++] = indices[e];
    indptr_r[i + 1] = (int32_t)mr;
  }
  counts[0] = n_tiles;
  counts[1] = mr;
  free(ek); free(row); free(in_tile); free(pair_count);
  return 0;
}

/*
 * Node relabelling for gather locality ("On Efficient Scaling of GNNs via
 * IO-Aware Layers Implementations", zh/ko technical summaries,
 * "Methodology" and results: graph reordering, which the pages find helps
 * neighbour-parallel (gather-dominated) kernels on high-degree graphs).  The
 * pages name no method; two textbook ones are provided.  perm[new] = old.
 *   method 0, degree : nodes by decreasing total degree (in + out, every
 *                      edge counted), ties by increasing id.
 *   method 1, RCM    : reverse Cuthill-McKee on the undirected simple graph
 *                      (j -> i and i -> j merged, self-loops and repeats
 *                      dropped).  While nodes are unvisited, the unvisited
 *                      node of least degree (smallest id on ties) starts a
 *                      breadth-first search that appends each dequeued
 *                      node's unvisited neighbours in increasing (degree, id)
 *                      order; the final order is reversed.
 * Returns 0, -1 for an unknown method, -2 on allocation failure.
 */
typedef struct { int64_t key; int32_t id; } orc_node_key;

static int orc_cmp_node(const void* a, const void* b) {
  const orc_node_key* x = (const orc_node_key*)a;
  const orc_node_key* y = (const orc_node_key*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return x->id < y->id ? -1 : (x->id > y->id ? 1 : 0);
}

static int orc_cmp_i32(const void* a, const void* b) {
  const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return x < y ? -1 : (x > y ? 1 : 0);
}

int oracle_reorder(int32_t N, int64_t M, const int32_t* indptr, const int32_t* indices,
                   int method, int32_t* perm) {
  if (method != 0 && method != 1) return -1;
  orc_node_key* nk = (orc_node_key*)malloc(((size_t)N + 1) * sizeof(orc_node_key));
  if (!nk) return -2;
  if (method == 0) {
    int64_t* deg = (int64_t*)calloc((size_t)N + 1, sizeof(int64_t));
    if (!deg) { free(nk); return -2; }
    for (int32_t i = 0; i < N; ++i) {
      deg[i] += indptr[i + 1] - indptr[i];
      for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) deg[indices[e]] += 1;
    }
    for (int32_t i = 0; i < N; ++i) { nk[i].key = -deg[i]; nk[i].id = i; }
    qsort(nk, (size_t)N, sizeof(orc_node_key), orc_cmp_node);
    for (int32_t i = 0; i < N; ++i) perm[i] = nk[i].id;
    free(deg);
    free(nk);
    return 0;
  }
  /* undirected simple adjacency: both directions, then sort + unique per node */
  int64_t* cnt = (int64_t*)calloc((size_t)N + 1, sizeof(int64_t));
  int64_t* start = (int64_t*)malloc(((size_t)N + 1) * sizeof(int64_t));
  int32_t* adj = (int32_t*)malloc((size_t)(2 * M > 0 ? 2 * M : 1) * sizeof(int32_t));
  int64_t* fill = (int64_t*)malloc(((size_t)N + 1) * sizeof(int64_t));
  int64_t* deg = (int64_t*)malloc(((size_t)N + 1) * sizeof(int64_t));
  unsigned char* seen = (unsigned char*)calloc((size_t)N + 1, 1);
  int32_t* order = (int32_t*)malloc(((size_t)N + 1) * sizeof(int32_t));
  orc_node_key* nb = (orc_node_key*)malloc(((size_t)N + 1) * sizeof(orc_node_key));
  if (!cnt || !start || !adj || !fill || !deg || !seen || !order || !nb) {
    free(nk); free(cnt); free(start); free(adj); free(fill); free(deg); free(seen); free(order);
    free(nb);
    return -2;
  }
  for (int32_t i = 0; i < N; ++i)
    for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e)
      if (indices[e] != i) { cnt[i] += 1; cnt[indices[e]] += 1; }
  start[0] = 0;
  for (int32_t i = 0; i < N; ++i) { start[i + 1] = start[i] + cnt[i]; fill[i] = start[i]; }
  for (int32_t i = 0; i < N; ++i)
    for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) {
      const int32_t j = indices[e];
      if (j == i) continue;
      adj[fill[i]++] = j;
      adj[fill[j]++] = i;
    }
  for (int32_t i = 0; i < N; ++i) {
    int32_t* a = adj + start[i];
    const int64_t n = start[i + 1] - start[i];
    qsort(a, (size_t)n, sizeof(int32_t), orc_cmp_i32);
    int64_t u = 0;
    for (int64_t k = 0; k < n; ++k)
      if (k == 0 || a[k] != a[k - 1]) a[u++] = a[k];
    deg[i] = u;
  }
  /* roots in (degree, id) order */
  for (int32_t i = 0; i < N; ++i) { nk[i].key = deg[i]; nk[i].id = i; }
  qsort(nk, (size_t)N, sizeof(orc_node_key), orc_cmp_node);
  int64_t head = 0, tail = 0, next_root = 0;
  while (tail < N) {
    while (seen[nk[next_root].id]) ++next_root;
    const int32_t r = nk[next_root].id;
    seen[r] = 1;
    order[tail++] = r;
    while (head < tail) {
      const int32_t v = order[head++];
      int64_t m = 0;
      for (int64_t k = 0; k < deg[v]; ++k) {
        const int32_t w = adj[start[v] + k];
        if (!seen[w]) { nb[m].key = deg[w]; nb[m].id = w; ++m; }
      }
      qsort(nb, (size_t)m, sizeof(orc_node_key), orc_cmp_node);
      for (int64_t k = 0; k < m; ++k) { seen[nb[k].id] = 1; order[tail++] = nb[k].id; }
    }
  }
  for (int32_t i = 0; i < N; ++i) perm[i] = order[N - 1 - i];
  free(nk); free(cnt); free(start); free(adj); free(fill); free(deg); free(seen); free(order);
  free(nb);
  return 0;
}

/*
 * The graph under a relabelling perm (perm[new] = old): row i of the result
 * is old row perm[i], its sources mapped to their new ids and sorted
 * ascending (repeated sources kept).
 */
int oracle_permute_csr(int32_t N, int64_t M, const int32_t* indptr, const int32_t* indices,
                       const int32_t* perm, int32_t* indptr_out, int32_t* indices_out) {
  int32_t* inv = (int32_t*)malloc(((size_t)N + 1) * sizeof(int32_t));
  if (!inv) return -2;
  for (int32_t i = 0; i < N; ++i) inv[perm[i]] = i;
  int64_t o = 0;
  indptr_out[0] = 0;
  for (int32_t i = 0; i < N; ++i) {
    const int32_t old = perm[i];
    const int64_t r0 = o;
    for (int64_t e = indptr[old]; e < indptr[old + 1]; ++e) indices_out[o++] = inv[indices[e]];
    qsort(indices_out + r0, (size_t)(o - r0), sizeof(int32_t), orc_cmp_i32);
    indptr_out[i + 1] = (int32_t)o;
  }
  (void)M;
  free(inv);
  return 0;
}

/*
 * Max / min pooling over the in-neighbours ("On Efficient Scaling of GNNs
 * via IO-Aware Layers Implementations", zh/ko technical summaries,
 * "Methodology", reduction-based layers: a per-edge message followed by a
 * reduction over the neighbourhood such as max or min pooling; here the
 * message of edge j -> i is the source row x[j]).
 *   op 0 (max) / 1 (min):
 *     out[r][f] = max (min) over the edges e of row r of x[col[e]][f]
 *     arg[r][f] = the smallest source id that attains it
 *   a row without edges gets out 0 and arg -1.
 * Backward of L = sum out * dout: dx[j][f] = sum of dout[r][f] over the rows
 * r with arg[r][f] == j (dx is [N, F] by node id, overwritten).
 * Row subsets work as for the attention oracle (row r is a row position).
 */
int oracle_reduce_forward(int64_t n_rows, const int64_t* row_ptr, const int32_t* col, int64_t F,
                          int op, const double* x, double* out, int32_t* arg) {
  if (op != 0 && op != 1) return -1;
  for (int64_t r = 0; r < n_rows; ++r) {
    for (int64_t f = 0; f < F; ++f) {
      double best = 0.0;
      int32_t who = -1;
      for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
        const int32_t j = col[e];
        const double v = x[(int64_t)j * F + f];
        const int better = who < 0 || (op == 0 ? v > best : v < best) || (v == best && j < who);
        if (better) { best = v; who = j; }
      }
      out[r * F + f] = best;
      arg[r * F + f] = who;
    }
  }
  return 0;
}

int oracle_reduce_backward(int64_t n_rows, int64_t N, int64_t F, const int32_t* arg,
                           const double* dout, double* dx) {
  memset(dx, 0, (size_t)(N * F) * sizeof(double));
  for (int64_t r = 0; r < n_rows; ++r)
    for (int64_t f = 0; f < F; ++f) {
      const int32_t j = arg[r * F + f];
      if (j >= 0) dx[(int64_t)j * F + f] += dout[r * F + f];
    }
  return 0;
}

/*
 * Sparse-dense product of the weighted adjacency with node features
 * ("On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
 * technical summaries, "Methodology", SpMM-based convolutions such as GCN:
 * H' = A H W, where the SpMM A H aggregates neighbour rows with the edge
 * weights): y[r][f] = sum over the edges e of row r of w[e] * x[col[e]][f].
 * A row without edges gets 0.  w holds one weight per edge in CSR order.
 */
int oracle_spmm(int64_t n_rows, const int64_t* row_ptr, const int32_t* col, const double* w,
                int64_t F, const double* x, double* y) {
  for (int64_t r = 0; r < n_rows; ++r) {
    double* yr = y + r * F;
    for (int64_t f = 0; f < F; ++f) yr[f] = 0.0;
    for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
      const double* xj = x + (int64_t)col[e] * F;
      for (int64_t f = 0; f < F; ++f) yr[f] += w[e] * xj[f];
    }
  }
  return 0;
}
