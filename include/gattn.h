/*
 * gattn.h -- C ABI of the fused CSR graph-attention engine for GB300 (sm_103a).
 *
 * The operation ("On Efficient Scaling of GNNs via IO-Aware Layers
 * Implementations", zh/ko technical summaries, section "Methodology",
 * attention-based layers): for every destination node i of a graph given in
 * CSR form (row i lists the sources j of the edges j -> i), score each
 * in-neighbour j, normalise the scores with a softmax over the neighbourhood
 * and sum the neighbours' values with those weights -- in one streaming pass
 * with an online softmax whose running max and sum stay in registers, so no
 * O(M*H) edge tensor is ever stored.  Only a per-node, per-head log-sum-exp
 * is kept; the backward pass recomputes the weights from it.  The graph
 * metadata (degree split, heavy-node edge chunks, transposed adjacency) is
 * built once per graph and cached ("Methodology", SpMM and reduction layers).
 *
 * Two score functions (the two attention layers the pages name):
 *   GATTN_SCORE_DOT   : s_ijh = scale * sum_d Q[i,h,d] K[j,h,d]
 *                       (Graph Transformer; scale = 1/sqrt(D) by default)
 *   GATTN_SCORE_GATV2 : s_ijh = sum_d a[h,d] * LeakyReLU(Q[i,h,d] + K[j,h,d])
 *                       (GATv2 with Q = x_l, K = x_r, slope 0.2 by default)
 * Then, for a node with at least one in-edge,
 *   alpha_ijh = exp(s_ijh - lse[i,h]),  lse[i,h] = log sum_j exp(s_ijh),
 *   out[i,h,:] = sum_j alpha_ijh V[j,h,:].
 * A node with no in-edges gets out = 0 and lse = -inf.
 *
 * Conventions shared by every entry point
 *   - Dense tensors (Q, K, V, out, dout, dQ, dK, dV) are row-major
 *     [N, H, D], contiguous, in the I/O dtype (fp32 or bf16); the base
 *     address must be 16-byte aligned.  lse is fp32 [N, H].  a and da are
 *     fp32 [H, D].
 *   - The graph is int32 CSR by destination: indptr[N+1] (indptr[0] = 0,
 *     non-decreasing, indptr[N] = M) and indices[M] (sources, in [0, N)).
 *     Rows need not be sorted; multi-edges are kept as separate edges.
 *   - Every pointer argument that names tensor data is a DEVICE pointer
 *     unless the argument's comment says "host".  All device memory is owned
 *     by the caller, except the plan's own buffers.
 *   - Calls are asynchronous on the given stream unless stated otherwise;
 *     a status other than GATTN_OK leaves outputs undefined.  No call aborts
 *     or traps; gattn_last_error() gives a message for the calling thread.
 *   - Supported head layouts: D a power of two with D * sizeof(dtype) in
 *     [16, 512] bytes, H a power of two, and H * D * sizeof(dtype) in
 *     [32, 2048] bytes.  Other shapes return GATTN_ERR_UNSUPPORTED.
 */
#ifndef GATTN_H_
#define GATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GATTN_API __attribute__((visibility("default")))
#else
#define GATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* gattn_stream_t;

typedef enum {
  GATTN_OK = 0,
  GATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, small workspace */
  GATTN_ERR_BAD_GRAPH = 2,   /* CSR violates the conventions above */
  GATTN_ERR_UNSUPPORTED = 3, /* (H, D, dtype) outside the supported set */
  GATTN_ERR_OOM = 4,         /* plan buffers could not be allocated */
  GATTN_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  GATTN_ERR_TIMEOUT = 6      /* a kernel gave up a bounded wait (see gattn_plan_check_errors) */
} gattn_status;

typedef enum { GATTN_F32 = 0, GATTN_BF16 = 1 } gattn_dtype;

typedef enum { GATTN_SCORE_DOT = 0, GATTN_SCORE_GATV2 = 1 } gattn_score_kind;

typedef enum { GATTN_REORDER_DEGREE = 0, GATTN_REORDER_RCM = 1 } gattn_reorder_kind;

typedef enum { GATTN_POOL_MAX = 0, GATTN_POOL_MIN = 1 } gattn_pool_op;

/* Score parameters.  Host struct; `a` is a device pointer. */
typedef struct {
  int32_t kind;    /* gattn_score_kind */
  float scale;     /* DOT: multiplier of q.k; 0 selects 1/sqrt(D) */
  const float* a;  /* GATV2: device fp32 [H, D]; ignored for DOT */
  float neg_slope; /* GATV2: LeakyReLU slope for z <= 0; use 0.2 for the usual layer */
} gattn_score;

/* Plan options.  Host struct; pass NULL for the defaults. */
typedef struct {
  int32_t heavy_threshold; /* node is heavy when its degree > this (max 256); <= 0: chosen
                              from the graph size, a power of two in [32, 256] */
  int32_t chunk;           /* edges per heavy-node chunk (max 256); <= 0: the threshold */
  int32_t tile_enable;     /* nonzero: also build the dense-tile split (needs N <= 2^23) */
  float tile_density;      /* a 128 x 128 block of (destination, source) ids with at least
                              ceil(tile_density * 16384) edges becomes a tile; <= 0: 1/16 */
} gattn_plan_opts;

/* Sizes of a built plan (host struct filled by gattn_plan_get_info). */
typedef struct {
  int32_t N;
  int64_t M;
  int32_t heavy_threshold;
  int32_t chunk;
  int64_t n_light;      /* destinations with degree <= threshold */
  int64_t n_heavy;      /* destinations with degree > threshold */
  int64_t n_chunks;     /* edge chunks of the heavy destinations */
  int64_t n_light_src;  /* sources with out-degree <= threshold */
  int64_t n_heavy_src;  /* sources with out-degree > threshold */
  int64_t n_src_chunks; /* edge chunks of the heavy sources (CSC) */
  int32_t max_deg;
  int32_t max_outdeg;
  size_t device_bytes;  /* device memory held by the plan */
  int64_t n_tiles;      /* dense tiles (0 unless tile_enable) */
  int64_t n_tile_rows;  /* 128-node row blocks that have tiles */
  int64_t tile_edges;   /* edges covered by the tiles' masks */
  int32_t tile_min_edges; /* edges that made a block a tile */
} gattn_plan_info;

typedef struct gattn_plan gattn_plan;

/*
 * Build the per-graph plan ("Methodology": degree-aware light/heavy split of
 * the nodes by a degree threshold, heavy nodes cut into edge chunks; the
 * transposed adjacency cached for the backward pass).
 *   indptr, indices : device int32 CSR (read during the call, not retained).
 *   N >= 0, M >= 0  : node and edge counts (M < 2^31).
 *   opts            : host, nullable.
 *   out             : host; receives the plan, which owns its device buffers.
 * The CSR is validated on the device first; a violation returns
 * GATTN_ERR_BAD_GRAPH.  Synchronises `stream` (sizes are read back).
 */
GATTN_API gattn_status gattn_plan_create(const int32_t* indptr, const int32_t* indices, int32_t N,
                               int64_t M, const gattn_plan_opts* opts, gattn_stream_t stream,
                               gattn_plan** out);

/* Free the plan's device buffers (synchronises the device first).  NULL is a no-op. */
GATTN_API gattn_status gattn_plan_destroy(gattn_plan* plan);

/* Host query of the plan's sizes. */
GATTN_API gattn_status gattn_plan_get_info(const gattn_plan* plan, gattn_plan_info* info);

/*
 * Copy the plan's integer metadata to HOST buffers (each nullable; sizes in
 * elements from gattn_plan_get_info).  Synchronous.  Definitions:
 *   deg[N], hist[33]      : in-degrees; hist[b] counts nodes of degree bin b
 *                           (bin 0: degree 0; bin b >= 1: 2^(b-1) <= deg < 2^b)
 *   light[n_light]        : ascending destinations with deg <= threshold
 *   chunks[3*n_chunks]    : (node, e0, e1) for heavy destinations in
 *                           ascending order, e0 = indptr[i] + k*chunk,
 *                           e1 = min(e0 + chunk, indptr[i+1])
 *   indptrT[N+1], csc_dst[M], csc_eid[M] : the transpose, edges stably
 *                           sorted by source over CSR edge order
 *   outdeg[N], hist_out[33], light_src[n_light_src], src_chunks[3*n_src_chunks]
 *                         : the same partition applied to the transpose
 */
GATTN_API gattn_status gattn_plan_export(const gattn_plan* plan, int32_t* deg, int32_t* hist,
                               int32_t* light, int32_t* chunks, int32_t* indptrT,
                               int32_t* csc_dst, int32_t* csc_eid, int32_t* outdeg,
                               int32_t* hist_out, int32_t* light_src, int32_t* src_chunks);

/*
 * Copy the dense-tile split to HOST buffers (each nullable; synchronous).
 * Nodes are cut into blocks of 128 ids; the block (rb, cb) holds the edges
 * j -> i with i / 128 == rb, j / 128 == cb.  A block with at least
 * tile_min_edges edges is a tile; tiles are listed in (rb, cb) order.
 *   tile_rb[n_tiles], tile_cb[n_tiles]
 *   masks[n_tiles * 512] : per tile 128 rows of 4 words; bit b of word w of
 *                          row r is set when the pair (i = 128 rb + r,
 *                          j = 128 cb + 32 w + b) occurs exactly once
 *   indptr_r[N+1], indices_r[M - tile_edges] : the residual CSR, every edge
 *                          not covered by a mask bit, in CSR order
 * Returns GATTN_ERR_INVALID_ARG for a plan built without tile_enable.
 */
GATTN_API gattn_status gattn_plan_export_tiles(const gattn_plan* plan, int32_t* tile_rb,
                                               int32_t* tile_cb, uint32_t* masks,
                                               int32_t* indptr_r, int32_t* indices_r);

/*
 * Copy the structures the tile backward walks to HOST buffers (each
 * nullable; synchronous; "Methodology", attention-based layers: the
 * backward recomputes the weights tile by tile, and the transposed adjacency
 * is cached for the source-side gradients).
 *   n_tcols (out)        : column blocks that have tiles
 *   tcol_cb[n_tcols]     : those column blocks, ascending
 *   tcol_ptr[n_tcols+1], tcol_tile[n_tiles] : tile ids of each column block,
 *                          ascending (so ascending row block)
 *   masks_t[n_tiles * 512] : the masks transposed: per tile 128 columns of 4
 *                          words; bit b of word w of column c is the mask bit
 *                          of row 32 w + b, column c
 *   indptrT_r[N+1], csc_dst_r[M - tile_edges] : the transpose of the
 *                          residual CSR, each column in residual CSR order
 * Call once with only n_tcols to size tcol_cb and tcol_ptr.  Returns
 * GATTN_ERR_INVALID_ARG for a plan built without tile_enable.
 */
GATTN_API gattn_status gattn_plan_export_tile_bwd(const gattn_plan* plan, int64_t* n_tcols,
                                                  int32_t* tcol_cb, int32_t* tcol_ptr,
                                                  int32_t* tcol_tile, uint32_t* masks_t,
                                                  int32_t* indptrT_r, int32_t* csc_dst_r);

/*
 * Synchronise the device and report whether any kernel run with this plan
 * since the last check gave up a bounded wait for its asynchronous copies
 * (every wait in the kernels has an iteration limit; on expiry the kernel
 * records the failure, waits -- again bounded -- for the copies it had
 * already issued, and returns instead of hanging; its outputs are then
 * undefined).  Returns GATTN_OK or GATTN_ERR_TIMEOUT.  On GATTN_ERR_TIMEOUT
 * it also clears the record and the plan's merge-tree arrival counters (a
 * warp that gave up may have left a count behind), so the plan can be used
 * again.  Synchronous.
 */
GATTN_API gattn_status gattn_plan_check_errors(const gattn_plan* plan);

/*
 * Test hook for the failure path above (not part of the method).  With
 * fail_first_wait nonzero, every warp of the attention passes run with this
 * plan (gattn_fwd's CSR pass, gattn_bwd_dq, gattn_bwd_dkdv, and the same
 * passes inside gattn_bwd and gattn_fwd_noalloc) treats its first wait for
 * gathered rows as expired without polling: it records the failure, waits
 * with the normal limit for every copy it had issued, and returns, so the
 * next gattn_plan_check_errors returns GATTN_ERR_TIMEOUT.  Zero restores
 * normal operation.  Host call; affects launches made after it.
 */
GATTN_API gattn_status gattn_plan_set_wait_test(gattn_plan* plan, int32_t fail_first_wait);

/*
 * Bytes of caller-owned device workspace that gattn_fwd / gattn_bwd need
 * for this plan and head layout (heavy-chunk partials, the backward's
 * per-node (lse, Delta) rows, GATv2 da partials).  Host call, no device work.
 */
GATTN_API gattn_status gattn_workspace_size(const gattn_plan* plan, int32_t H, int32_t D,
                                  gattn_dtype dtype, size_t* bytes);

/*
 * Workspace ownership.  In the call signatures of the method's contract
 * the plan owns its scratch (heavy-chunk partials, the per-node Delta); here
 * the caller passes it to gattn_fwd and gattn_bwd as `workspace`, sized by
 * gattn_workspace_size.  The scratch depends on the head layout (H, D) of
 * each call, which the plan does not know, and caller-owned memory lets one
 * framework allocator (e.g. PyTorch's caching allocator) hold every buffer.
 * Either way the forward and backward calls allocate nothing.
 *
 * Forward ("Methodology", attention-based layers, forward pass): one
 * streaming pass over each destination's in-neighbours with an online
 * softmax; heavy destinations are split over edge chunks whose partial
 * (max, sum, acc) triples are merged in chunk order.
 *   Q, K, V   : device [N, H, D] in `dtype` (GATv2: Q = x_l, K = x_r).
 *   score     : host struct (see gattn_score).
 *   out       : device [N, H, D] in `dtype` (written).
 *   lse       : device fp32 [N, H] (written; natural log; -inf for isolated nodes).
 *   workspace : device, >= gattn_workspace_size bytes, 16-byte aligned;
 *               its contents need no initialisation.
 * Calls that share a plan or a workspace must not overlap on the device.
 * With a plan built with tile_enable, the DOT score, bf16 and D = 64 or
 * 128, the forward runs in two launches ("Methodology", attention-based
 * layers, tensor-core optimisation): the CSR pass over the residual edges,
 * then the tiles on the tensor cores, merged per node; otherwise the CSR
 * pass covers every edge.  Both give the same softmax attention.
 */
GATTN_API gattn_status gattn_fwd(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                       const void* Q, const void* K, const void* V, const gattn_score* score,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       gattn_stream_t stream);

/*
 * Backward ("Methodology", attention-based layers, backward pass): the
 * attention weights are recomputed on the fly from the cached lse; dQ is
 * gathered over the CSR, dK and dV over the cached transpose.
 *   Q, K, V, out, lse : as passed to / produced by gattn_fwd with this plan.
 *   dout      : device [N, H, D] in `dtype`, gradient of the loss w.r.t. out.
 *   dQ, dK, dV: device [N, H, D] in `dtype` (written, not accumulated).
 *   da        : GATv2: device fp32 [H, D] (written), or NULL to skip; DOT: ignored.
 *   workspace : as for gattn_fwd.
 * With a plan built with tile_enable, the DOT score, bf16 and D = 64 or
 * 128, each pass runs in two launches: the CSR (CSC) pass over the
 * residual edges, then the tiles on the tensor cores, which recompute their
 * score blocks and add their dQ (dK and dV) to the rows the first launch
 * wrote; otherwise the passes cover every edge.
 */
GATTN_API gattn_status gattn_bwd(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                       const void* Q, const void* K, const void* V, const gattn_score* score,
                       const void* out, const void* dout, const float* lse, void* dQ, void* dK,
                       void* dV, float* da, void* workspace, size_t workspace_bytes,
                       gattn_stream_t stream);

/*
 * The two passes of gattn_bwd as separate calls (gattn_bwd = dq then dkdv on
 * one stream).  gattn_bwd_dq runs the CSR pass: writes dQ, da (GATv2,
 * nullable) and the per-node Delta = dout . out into the workspace.
 * gattn_bwd_dkdv runs the CSC pass: writes dK, dV and reads that Delta, so
 * it must follow a gattn_bwd_dq with the same plan, inputs and workspace.
 */
GATTN_API gattn_status gattn_bwd_dq(const gattn_plan* plan, int32_t H, int32_t D,
                                    gattn_dtype dtype, const void* Q, const void* K,
                                    const void* V, const gattn_score* score, const void* out,
                                    const void* dout, const float* lse, void* dQ, float* da,
                                    void* workspace, size_t workspace_bytes,
                                    gattn_stream_t stream);
GATTN_API gattn_status gattn_bwd_dkdv(const gattn_plan* plan, int32_t H, int32_t D,
                                      gattn_dtype dtype, const void* Q, const void* K,
                                      const void* V, const gattn_score* score, const void* dout,
                                      const float* lse, void* dK, void* dV, void* workspace,
                                      size_t workspace_bytes, gattn_stream_t stream);

/*
 * gattn_fwd without a workspace argument, for callers that cannot allocate
 * device memory where they run the layer: code under a memory pool or
 * allocator it does not own, or a plugin host that hands over only the
 * input and output tensors.  The paper has no counterpart to this call.
 * Same arguments as gattn_fwd minus the workspace; the heavy-chunk scratch
 * comes from one fixed 32 MiB array compiled into the library, so the call
 * allocates nothing.
 *   - It always runs the CSR pass over every edge.  On a plan built without
 *     tile_enable its results equal gattn_fwd's bit for bit; on a tiled plan
 *     (where gattn_fwd may run the dense tiles on the tensor cores) they
 *     agree with gattn_fwd within the rounding tolerance, not exactly.
 *   - A plan and head layout whose scratch would exceed 32 MiB are rejected
 *     with GATTN_ERR_INVALID_ARG (use gattn_fwd with a workspace instead),
 *     as are a null or misaligned tensor, lse or (GATv2) a pointer.
 *   - The first call in a CUDA context (per device, and again after the
 *     context is replaced, e.g. by cudaDeviceReset) looks up the array's
 *     device address with cudaGetSymbolAddress and caches it; make that
 *     first call before any stream capture begins.
 *   - All calls share the array, which keeps whatever the last call left in
 *     it (nothing in it needs to start at zero): calls whose kernels may
 *     overlap on the GPU (different streams or host threads) race and must
 *     be ordered.
 *   - The array lives on every device that loads the library until exit.
 */
GATTN_API gattn_status gattn_fwd_noalloc(const gattn_plan* plan, int32_t H, int32_t D,
                                         gattn_dtype dtype, const void* Q, const void* K,
                                         const void* V, const gattn_score* score, void* out,
                                         float* lse, gattn_stream_t stream);

/* Message of the last failing call on this thread ("" if none).  Never NULL. */
GATTN_API const char* gattn_last_error(void);

/* Library version string, e.g. "gattn 0.1.0 sm_103a". */
GATTN_API const char* gattn_version(void);

/*
 * Max / min pooling over the in-neighbours ("Methodology", reduction-based
 * layers: a per-edge message -- here the source row -- reduced over the
 * neighbourhood; light nodes in one pass, heavy nodes over edge chunks merged
 * by atomics on packed (value, index) pairs), on the same plan.
 *   x[N, F], out[N, F] : device, I/O dtype; F * sizeof(dtype) a power of two
 *                        in [32, 2048] bytes (else GATTN_ERR_UNSUPPORTED).
 *   op                 : GATTN_POOL_MAX or GATTN_POOL_MIN.
 *   out[i][f] = max (min) over the sources j of i of x[j][f] (exact: a copy of
 *   an input value); arg[i][f] (device int32 [N, F]) = the smallest such j;
 *   a node without in-edges gets out 0 and arg -1.  NaN inputs are not
 *   supported.
 *   workspace          : device, gattn_pool_workspace_size bytes, 16-byte
 *                        aligned; cleared by the calls themselves.
 * Backward: dx[j][f] = sum of dout[i][f] over the nodes i with arg[i][f] == j
 * (fp32 accumulation in the workspace, rounded once to the I/O dtype; the
 * order of the additions is not fixed, so the last bits may vary between
 * runs).  Asynchronous on `stream`.
 */
GATTN_API gattn_status gattn_pool_workspace_size(const gattn_plan* plan, int32_t F,
                                                 gattn_dtype dtype, size_t* bytes);
GATTN_API gattn_status gattn_pool_fwd(const gattn_plan* plan, int32_t F, gattn_dtype dtype,
                                      int32_t op, const void* x, void* out, int32_t* arg,
                                      void* workspace, size_t workspace_bytes,
                                      gattn_stream_t stream);
GATTN_API gattn_status gattn_pool_bwd(const gattn_plan* plan, int32_t F, gattn_dtype dtype,
                                      const int32_t* arg, const void* dout, void* dx,
                                      void* workspace, size_t workspace_bytes,
                                      gattn_stream_t stream);

/*
 * Weighted SpMM with the adjacency ("Methodology", SpMM-based convolutions
 * such as GCN: H' = A H W; the transposed adjacency is cached for the
 * backward; a weighted block-sparse form of locally dense neighbourhoods
 * runs on the tensor cores), on the same plan:
 *   transpose = 0 : y[i] = sum over the edges e = (j -> i) of w[e] x[j]
 *   transpose = 1 : y[j] = sum over the edges e = (j -> i) of w[e] x[i]
 *                   (the backward of the first: dX = A^T dY)
 *   w      : device fp32 [M], one weight per edge in the plan's CSR order.
 *   x, y   : device [N, F] in `dtype`, distinct; F * sizeof(dtype) a power of
 *            two in [32, 2048] bytes.  A node without edges gets 0.
 * With transpose = 0, a plan built with tile_enable, bf16 and F a multiple
 * of 64, the tiles' edges run as bf16-weight [128 x 128] x [128 x F] tensor-
 * core products added to the CSR result of the other edges (weights rounded
 * to bf16 there, and that CSR part rounded to bf16 before the addition);
 * otherwise every edge goes through the CSR pass (fp32 sums, one rounding).
 *   workspace : device, gattn_spmm_workspace_size bytes, 16-byte aligned.
 */
GATTN_API gattn_status gattn_spmm_workspace_size(const gattn_plan* plan, int32_t F,
                                                 gattn_dtype dtype, size_t* bytes);
GATTN_API gattn_status gattn_spmm(const gattn_plan* plan, int32_t F, gattn_dtype dtype,
                                  const float* w, const void* x, void* y, int32_t transpose,
                                  void* workspace, size_t workspace_bytes, gattn_stream_t stream);

/*
 * Node relabelling for gather locality ("Methodology" and results: graph
 * reordering helps gather-dominated kernels on high-degree graphs; the
 * pages name no method).  HOST pointers, synchronous, no device work.
 *   kind GATTN_REORDER_DEGREE : nodes by decreasing total degree (in + out,
 *        every edge counted), ties by increasing id.
 *   kind GATTN_REORDER_RCM    : reverse Cuthill-McKee on the undirected
 *        simple graph (j -> i and i -> j merged, self-loops and repeats
 *        dropped): while nodes are unvisited, the unvisited node of least
 *        degree (smallest id on ties) roots a breadth-first search that
 *        appends each dequeued node's unvisited neighbours in increasing
 *        (degree, id) order; the final order is reversed.
 *   perm[N] : receives perm[new id] = old id.
 * Returns GATTN_ERR_BAD_GRAPH for an invalid CSR.
 */
GATTN_API gattn_status gattn_reorder(const int32_t* indptr, const int32_t* indices, int32_t N,
                                     int64_t M, int32_t kind, int32_t* perm);

/*
 * The graph under a relabelling (HOST pointers, synchronous): row i of the
 * output is old row perm[i], its sources renamed to their new ids and sorted
 * ascending (repeated sources kept).  indptr_out[N+1], indices_out[M].
 * Returns GATTN_ERR_INVALID_ARG when perm is not a permutation of [0, N).
 */
GATTN_API gattn_status gattn_permute_csr(const int32_t* indptr, const int32_t* indices,
                                         int32_t N, int64_t M, const int32_t* perm,
                                         int32_t* indptr_out, int32_t* indices_out);

/*
 * Permute the rows of a dense device tensor of N rows of row_bytes bytes (a
 * multiple of 16; src and dst distinct, 16-byte aligned device pointers;
 * perm a device int32 permutation of [0, N)): inverse = 0 gathers, dst row i
 * = src row perm[i] (features into the new labelling); inverse = 1
 * scatters, dst row perm[i] = src row i (results back to the old one).
 * Asynchronous on `stream`; entries of perm outside [0, N) are skipped.
 */
GATTN_API gattn_status gattn_permute_rows(const void* src, void* dst, const int32_t* perm,
                                          int32_t N, int64_t row_bytes, int32_t inverse,
                                          gattn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GATTN_H_ */
