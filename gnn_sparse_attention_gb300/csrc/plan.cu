// plan.cu -- per-graph plan builder, entirely on the device.
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology": nodes are split by a degree threshold
// into light and heavy sets and heavy nodes are tiled over edge chunks
// (reduction layers); graph metadata and the transposed adjacency are built
// once and cached for the backward pass (SpMM layers).  Here the same split
// drives the attention kernels on both the CSR (destinations) and the cached
// CSC (sources).
//
// Steps: validate the CSR -> degrees, histograms and split flags -> integer
// exclusive scans -> item lists -> CSC by a stable LSD radix sort of the
// edge ids keyed by source (so each column lists its edges in CSR order).
// Every result is integer and independent of thread scheduling.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gattn_internal.cuh"

namespace gattn {

namespace {

constexpr int kScanItems = 8;
constexpr int kTile = kThreads * kScanItems;  // 2048 elements per scan / sort tile

#define GATTN_CUDA(call)                                                              \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess) {                                                          \
      set_error("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__,     \
                __LINE__);                                                            \
      return e_ == cudaErrorMemoryAllocation ? GATTN_ERR_OOM : GATTN_ERR_CUDA;        \
    }                                                                                 \
  } while (0)

// ---------------------------------------------------------------------------
// validation: bit 1 indptr[0] != 0, bit 2 indptr[N] != M, bit 4 decreasing
// indptr, bit 8 a source outside [0, N)
// ---------------------------------------------------------------------------
__global__ void k_validate(const int32_t* __restrict__ indptr, const int32_t* __restrict__ indices,
                           int32_t N, int64_t M, int32_t* err) {
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int bad = 0;
  if (tid == 0) {
    if (indptr[0] != 0) bad |= 1;
    if ((int64_t)indptr[N] != M) bad |= 2;
  }
  for (int64_t i = tid; i < N; i += stride)
    if (indptr[i + 1] < indptr[i]) bad |= 4;
  for (int64_t e = tid; e < M; e += stride) {
    const int32_t j = indices[e];
    if (j < 0 || j >= N) bad |= 8;
  }
  if (bad) atomicOr(err, bad);
}

__device__ __forceinline__ int degree_bin(int32_t d) { return d <= 0 ? 0 : 32 - __clz(d); }

// Degrees from a row pointer, histogram, max, and the split counts:
// light[i] = deg <= T, heavy[i] = deg > T, nchunk[i] = heavy ? ceil(deg/C) : 0.
// Arrays light/heavy/nchunk have N+1 entries, the last one 0 (scan totals).
__global__ void k_degrees(const int32_t* __restrict__ ptr, int32_t N, int32_t T, int32_t C,
                          int32_t* __restrict__ deg, int32_t* __restrict__ hist,
                          int32_t* __restrict__ maxdeg, int32_t* __restrict__ light,
                          int32_t* __restrict__ heavy, int32_t* __restrict__ nchunk) {
  __shared__ int32_t s_hist[33];
  __shared__ int32_t s_max;
  if (threadIdx.x < 33) s_hist[threadIdx.x] = 0;
  if (threadIdx.x == 0) s_max = 0;
  __syncthreads();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int32_t my_max = 0;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i <= N; i += stride) {
    if (i == N) {
      light[N] = heavy[N] = nchunk[N] = 0;
      continue;
    }
    const int32_t d = ptr[i + 1] - ptr[i];
    deg[i] = d;
    atomicAdd(&s_hist[degree_bin(d)], 1);
    my_max = max(my_max, d);
    const bool h = d > T;
    light[i] = h ? 0 : 1;
    heavy[i] = h ? 1 : 0;
    nchunk[i] = h ? (d + C - 1) / C : 0;
  }
  atomicMax(&s_max, my_max);
  __syncthreads();
  if (threadIdx.x < 33 && s_hist[threadIdx.x]) atomicAdd(&hist[threadIdx.x], s_hist[threadIdx.x]);
  if (threadIdx.x == 0) atomicMax(maxdeg, s_max);
}

__global__ void k_count_sources(const int32_t* __restrict__ indices, int64_t M,
                                int32_t* __restrict__ outdeg) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < M; e += stride)
    atomicAdd(&outdeg[indices[e]], 1);
}

// Row pointer from counts: ptr[i] = exclusive scan (computed separately).
// Item lists: chunks of heavy rows first (item index = chunk index, w =
// heavy id), then light rows (w = -1).  Also the exported light / chunk
// arrays and hfirst (first chunk of every heavy row, plus the total).
__global__ void k_fill_items(const int32_t* __restrict__ ptr, int32_t N, int32_t C,
                             const int32_t* __restrict__ light_pos,
                             const int32_t* __restrict__ heavy_pos,
                             const int32_t* __restrict__ chunk_pos, int64_t n_chunks,
                             int64_t n_heavy, int32_t* __restrict__ light_list,
                             int4* __restrict__ items, int32_t* __restrict__ hfirst) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < N; i += stride) {
    const int32_t e0 = ptr[i], e1 = ptr[i + 1];
    const int32_t lp = light_pos[i];
    if (light_pos[i + 1] != lp) {  // light row
      light_list[lp] = (int32_t)i;
      items[n_chunks + lp] = make_int4((int)i, e0, e1, -1);
    } else {
      const int32_t h = heavy_pos[i];
      int32_t c = chunk_pos[i];
      hfirst[h] = c;
      for (int32_t s = e0; s < e1; s += C, ++c)
        items[c] = make_int4((int)i, s, min(s + C, e1), h);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) hfirst[n_heavy] = (int32_t)n_chunks;
}

// Item edge counts (for the unit segmentation).
// Merge trees over the chunks of every heavy node (fan-in kTreeFanIn).
__device__ __forceinline__ int32_t tree_inner(int32_t n) {
  int32_t total = 0;
  while (n > 1) {
    n = (n + kTreeFanIn - 1) / kTreeFanIn;
    total += n;
  }
  return total;
}

__global__ void k_tree_sizes(const int32_t* __restrict__ hfirst, int64_t n_heavy,
                             int32_t* __restrict__ inner) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t h = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; h <= n_heavy; h += stride)
    inner[h] = h < n_heavy ? tree_inner(hfirst[h + 1] - hfirst[h]) : 0;
}

// One thread per heavy node builds its tree level by level: the children of
// inner node p of a level are consecutive slots of the level below.
__global__ void k_tree_fill(const int32_t* __restrict__ hfirst, int64_t n_heavy, int64_t n_chunks,
                            const int32_t* __restrict__ inner_pos, int32_t* __restrict__ parent,
                            int2* __restrict__ kids) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t h = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; h < n_heavy; h += stride) {
    int32_t lo = hfirst[h], n = hfirst[h + 1] - hfirst[h];
    int32_t next = (int32_t)n_chunks + inner_pos[h];  // next free inner slot
    if (n == 1) parent[lo] = -1;
    while (n > 1) {
      const int32_t m = (n + kTreeFanIn - 1) / kTreeFanIn;
      for (int32_t q = 0; q < m; ++q) {
        const int32_t c0 = lo + q * kTreeFanIn;
        const int32_t cn = min(kTreeFanIn, n - q * kTreeFanIn);
        kids[next + q - n_chunks] = make_int2(c0, cn);
        for (int32_t c = 0; c < cn; ++c) parent[c0 + c] = next + q;
      }
      if (m == 1) parent[next] = -1;
      lo = next;
      next += m;
      n = m;
    }
  }
}

// Degree binning of the work items: key = kMaxItemEdges - edge count, so a
// stable ascending sort lists items by decreasing length, ties in item order.
__global__ void k_length_keys(const int4* __restrict__ items, int64_t n, int32_t* __restrict__ key,
                              int32_t* __restrict__ val) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    key[i] = kMaxItemEdges - (items[i].z - items[i].y);
    val[i] = (int32_t)i;
  }
}

__global__ void k_gather_sorted(const int4* __restrict__ items, const int32_t* __restrict__ order,
                                int64_t n, int4* __restrict__ sorted) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int32_t it = order[i];
    const int4 x = items[it];
    sorted[i] = make_int4(x.x, x.y, x.z, it);
  }
}

// ---------------------------------------------------------------------------
// exclusive scan of int32 (tiles of 2048, recursive over tile totals)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* s_warp,
                                                        int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < kWarpsPerBlock ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < kWarpsPerBlock; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarpsPerBlock) s_warp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int32_t before = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[kWarpsPerBlock - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void k_scan_tiles(const int32_t* __restrict__ in, int32_t* __restrict__ out, int64_t n,
                             int32_t* __restrict__ tile_sums) {
  __shared__ int32_t s_warp[kWarpsPerBlock];
  const int64_t base = int64_t(blockIdx.x) * kTile + int64_t(threadIdx.x) * kScanItems;
  int32_t v[kScanItems];
  int32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    v[k] = base + k < n ? in[base + k] : 0;
    sum += v[k];
  }
  int32_t total;
  int32_t run = block_exclusive_scan(sum, s_warp, &total);
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < n) out[base + k] = run;
    run += v[k];
  }
  if (threadIdx.x == 0 && tile_sums) tile_sums[blockIdx.x] = total;
}

__global__ void k_scan_add(int32_t* __restrict__ out, int64_t n, const int32_t* __restrict__ offs) {
  const int32_t add = offs[blockIdx.x];
  const int64_t base = int64_t(blockIdx.x) * kTile;
  for (int k = threadIdx.x; k < kTile; k += blockDim.x)
    if (base + k < n) out[base + k] += add;
}

struct Scratch {
  std::vector<void*> ptrs;
  ~Scratch() {
    for (void* p : ptrs) cudaFree(p);
  }
  template <typename T>
  cudaError_t get(T** p, size_t n) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, (n ? n : 1) * sizeof(T));
    if (e == cudaSuccess) ptrs.push_back(q);
    *p = reinterpret_cast<T*>(q);
    return e;
  }
};

gattn_status exclusive_scan(const int32_t* in, int32_t* out, int64_t n, Scratch& scr,
                            cudaStream_t st) {
  if (n <= 0) return GATTN_OK;
  const int64_t tiles = (n + kTile - 1) / kTile;
  if (tiles == 1) {
    k_scan_tiles<<<1, kThreads, 0, st>>>(in, out, n, nullptr);
    GATTN_CUDA(cudaGetLastError());
    return GATTN_OK;
  }
  int32_t *sums = nullptr, *offs = nullptr;
  GATTN_CUDA(scr.get(&sums, tiles));
  GATTN_CUDA(scr.get(&offs, tiles));
  k_scan_tiles<<<(unsigned)tiles, kThreads, 0, st>>>(in, out, n, sums);
  GATTN_CUDA(cudaGetLastError());
  gattn_status s = exclusive_scan(sums, offs, tiles, scr, st);
  if (s != GATTN_OK) return s;
  k_scan_add<<<(unsigned)tiles, kThreads, 0, st>>>(out, n, offs);
  GATTN_CUDA(cudaGetLastError());
  return GATTN_OK;
}

// ---------------------------------------------------------------------------
// stable LSD radix sort of (key = source, value = edge id), 8-bit digits
// ---------------------------------------------------------------------------
__global__ void k_radix_hist(const int32_t* __restrict__ keys, int64_t n, int shift,
                             int64_t n_tiles, int32_t* __restrict__ hist) {
  __shared__ int32_t s_cnt[256];
  s_cnt[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = int64_t(blockIdx.x) * kTile;
  for (int k = threadIdx.x; k < kTile; k += blockDim.x)
    if (base + k < n) atomicAdd(&s_cnt[(keys[base + k] >> shift) & 255], 1);
  __syncthreads();
  hist[int64_t(threadIdx.x) * n_tiles + blockIdx.x] = s_cnt[threadIdx.x];
}

// Elements of a tile are taken in rounds of 256 in index order; within a
// round, warp w's lanes precede warp w+1's, and lanes are ordered by index,
// so (previous rounds, earlier warps, lower lanes) is exactly "earlier in the
// input": the scatter is stable.
__global__ void k_radix_scatter(const int32_t* __restrict__ kin, const int32_t* __restrict__ vin,
                                int32_t* __restrict__ kout, int32_t* __restrict__ vout, int64_t n,
                                int shift, int64_t n_tiles, const int32_t* __restrict__ offs) {
  __shared__ int32_t s_wcnt[kWarpsPerBlock][256];
  __shared__ int32_t s_woff[kWarpsPerBlock][256];
  __shared__ int32_t s_base[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int w = 0; w < kWarpsPerBlock; ++w) s_wcnt[w][threadIdx.x] = 0;
  s_base[threadIdx.x] = offs[int64_t(threadIdx.x) * n_tiles + blockIdx.x];
  __syncthreads();
  const int64_t base = int64_t(blockIdx.x) * kTile;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < kScanItems; ++r) {
    const int64_t idx = base + int64_t(r) * kThreads + threadIdx.x;
    const bool valid = idx < n;
    const int32_t key = valid ? kin[idx] : 0;
    const int32_t val = valid ? vin[idx] : 0;
    const int d = valid ? ((key >> shift) & 255) : 256;
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const int rank = __popc(peers & lt_mask);
    if (valid && rank == 0) s_wcnt[warp][d] = __popc(peers);
    __syncthreads();
    {
      const int dig = threadIdx.x;
      int32_t acc = s_base[dig];
      for (int w = 0; w < kWarpsPerBlock; ++w) {
        const int32_t c = s_wcnt[w][dig];
        s_woff[w][dig] = acc;
        acc += c;
        s_wcnt[w][dig] = 0;
      }
      s_base[dig] = acc;
    }
    __syncthreads();
    if (valid) {
      const int32_t pos = s_woff[warp][d] + rank;
      kout[pos] = key;
      vout[pos] = val;
    }
  }
}

__global__ void k_iota(int32_t* __restrict__ v, int64_t n) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    v[i] = (int32_t)i;
}

// csc_dst[p] = destination row of CSR edge csc_eid[p] (last i with indptr[i] <= e)
__global__ void k_edge_rows(const int32_t* __restrict__ indptr, int32_t N,
                            const int32_t* __restrict__ eid, int64_t M, int32_t* __restrict__ dst) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; p < M; p += stride) {
    const int32_t e = eid[p];
    int32_t lo = 0, hi = N;  // invariant: indptr[lo] <= e < indptr[hi]
    while (hi - lo > 1) {
      const int32_t mid = lo + (hi - lo) / 2;
      if (indptr[mid] <= e) lo = mid;
      else hi = mid;
    }
    dst[p] = lo;
  }
}

// ---------------------------------------------------------------------------
// dense tiles ("Methodology", attention-based layers, tensor-core
// optimisation: locally dense neighbourhoods packed into block tiles)
// ---------------------------------------------------------------------------
// Block key of every edge, (row block) * nb + (column block) as an unsigned
// bit pattern, the edge id, and the edge's row for the mask pass.
__global__ void k_block_keys(const int32_t* __restrict__ indptr, int32_t N,
                             const int32_t* __restrict__ indices, int64_t M, uint32_t nb,
                             int32_t* __restrict__ key, int32_t* __restrict__ eid,
                             int32_t* __restrict__ row) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < M; e += stride) {
    int32_t lo = 0, hi = N;  // invariant: indptr[lo] <= e < indptr[hi]
    while (hi - lo > 1) {
      const int32_t mid = lo + (hi - lo) / 2;
      if (indptr[mid] <= e) lo = mid;
      else hi = mid;
    }
    row[e] = lo;
    eid[e] = (int32_t)e;
    key[e] = (int32_t)(uint32_t(lo / kTileRows) * nb + uint32_t(indices[e] / kTileRows));
  }
}

// head[p] = 1 where the sorted keys start a new block (head[n] = 0)
__global__ void k_run_heads(const int32_t* __restrict__ key, int64_t n, int32_t* __restrict__ head) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i <= n; i += stride)
    head[i] = i < n && (i == 0 || key[i] != key[i - 1]) ? 1 : 0;
}

// start[pos[i]] = i at every head; start[n_runs] = n
__global__ void k_run_starts(const int32_t* __restrict__ head, const int32_t* __restrict__ pos,
                             int64_t n, int32_t* __restrict__ start) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i <= n; i += stride)
    if (i == n) start[pos[n]] = (int32_t)n;
    else if (head[i]) start[pos[i]] = (int32_t)i;
}

// dense[r] = 1 for runs (blocks) of at least tile_min edges (dense[n_runs] = 0)
__global__ void k_run_dense(const int32_t* __restrict__ start, int64_t n_runs, int32_t tile_min,
                            int32_t* __restrict__ dense) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r <= n_runs; r += stride)
    dense[r] = r < n_runs && start[r + 1] - start[r] >= tile_min ? 1 : 0;
}

__global__ void k_tile_meta(const int32_t* __restrict__ start, const int32_t* __restrict__ dense,
                            const int32_t* __restrict__ tpos, int64_t n_runs,
                            const int32_t* __restrict__ key, uint32_t nb,
                            int32_t* __restrict__ tile_rb, int32_t* __restrict__ tile_cb,
                            int32_t* __restrict__ tbeg, int32_t* __restrict__ tend) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r < n_runs; r += stride) {
    if (!dense[r]) continue;
    const int32_t t = tpos[r];
    const uint32_t k = uint32_t(key[start[r]]);
    tile_rb[t] = int32_t(k / nb);
    tile_cb[t] = int32_t(k % nb);
    tbeg[t] = start[r];
    tend[t] = start[r + 1];
  }
}

// One block per tile: set the bits of the tile's (row, column) pairs in
// shared memory, drop the pairs seen more than once, publish the mask and
// flag the edges it covers.
__global__ void k_tile_masks(const int32_t* __restrict__ tbeg, const int32_t* __restrict__ tend,
                             const int32_t* __restrict__ seid, const int32_t* __restrict__ row,
                             const int32_t* __restrict__ indices, uint32_t* __restrict__ mask,
                             uint8_t* __restrict__ in_tile, int32_t* __restrict__ slot) {
  __shared__ uint32_t s_seen[kTileRows * 4], s_dup[kTileRows * 4];
  const int64_t t = blockIdx.x;
  for (int w = threadIdx.x; w < kTileRows * 4; w += blockDim.x) s_seen[w] = s_dup[w] = 0;
  __syncthreads();
  const int32_t b = tbeg[t], e1 = tend[t];
  for (int32_t p = b + threadIdx.x; p < e1; p += blockDim.x) {
    const int32_t e = seid[p];
    const int r = row[e] % kTileRows, c = indices[e] % kTileRows;
    const uint32_t bit = 1u << (c % 32);
    if (atomicOr(&s_seen[r * 4 + c / 32], bit) & bit) atomicOr(&s_dup[r * 4 + c / 32], bit);
  }
  __syncthreads();
  for (int w = threadIdx.x; w < kTileRows * 4; w += blockDim.x) {
    const uint32_t m = s_seen[w] & ~s_dup[w];
    mask[t * kTileRows * 4 + w] = m;
    s_seen[w] = m;
  }
  __syncthreads();
  for (int32_t p = b + threadIdx.x; p < e1; p += blockDim.x) {
    const int32_t e = seid[p];
    const int r = row[e] % kTileRows, c = indices[e] % kTileRows;
    if ((s_seen[r * 4 + c / 32] >> (c % 32)) & 1u) {
      in_tile[e] = 1;
      const int64_t sl = t * kTileRows * kTileRows + r * kTileRows + c;
      if (sl < INT32_MAX) slot[e] = int32_t(sl);  // tiles beyond 2^31 weights: no WSB slot
    }
  }
}

// Residual CSR: a warp per row counts (then copies, in CSR order) the edges
// outside the tiles.
__global__ void k_res_count(const int32_t* __restrict__ indptr, int32_t N,
                            const uint8_t* __restrict__ in_tile, int32_t* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i <= N; i += warps) {
    if (i == N) {
      if (lane == 0) cnt[N] = 0;
      continue;
    }
    int32_t c = 0;
    for (int32_t e = indptr[i] + lane; e < indptr[i + 1]; e += 32) c += in_tile[e] ? 0 : 1;
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) cnt[i] = c;
  }
}

__global__ void k_res_fill(const int32_t* __restrict__ indptr, int32_t N,
                           const int32_t* __restrict__ indices, const uint8_t* __restrict__ in_tile,
                           const int32_t* __restrict__ ptr_r, int32_t* __restrict__ idx_r,
                           int32_t* __restrict__ eid_r) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < N; i += warps) {
    int32_t out = ptr_r[i];
    const int32_t e1 = indptr[i + 1];
    for (int32_t e0 = indptr[i]; e0 < e1; e0 += 32) {
      const int32_t e = e0 + lane;
      const bool keep = e < e1 && !in_tile[e];
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const int32_t o = out + __popc(bal & ((1u << lane) - 1u));
        idx_r[o] = indices[e];
        eid_r[o] = e;
      }
      out += __popc(bal);
    }
  }
}

// Row blocks that have tiles (tiles are in row-block order).
__global__ void k_trow_heads(const int32_t* __restrict__ tile_rb, int64_t n, int32_t* __restrict__ head) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t <= n; t += stride)
    head[t] = t < n && (t == 0 || tile_rb[t] != tile_rb[t - 1]) ? 1 : 0;
}

__global__ void k_trow_fill(const int32_t* __restrict__ tile_rb, const int32_t* __restrict__ head,
                            const int32_t* __restrict__ pos, int64_t n, int32_t* __restrict__ trow_rb,
                            int32_t* __restrict__ trow_ptr) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t <= n; t += stride)
    if (t == n) trow_ptr[pos[n]] = (int32_t)n;
    else if (head[t]) {
      trow_rb[pos[t]] = tile_rb[t];
      trow_ptr[pos[t]] = (int32_t)t;
    }
}

// Transposed tile masks: bit i % 128 of column j % 128 (4 words a column),
// for the backward pass that walks a tile by source column.  One block of
// 128 threads per tile; thread j assembles column j.
__global__ void k_mask_transpose(const uint32_t* __restrict__ mask, uint32_t* __restrict__ mask_t) {
  __shared__ uint32_t s_m[kTileRows * 4];
  const int64_t base = int64_t(blockIdx.x) * kTileRows * 4;
  for (int w = threadIdx.x; w < kTileRows * 4; w += blockDim.x) s_m[w] = mask[base + w];
  __syncthreads();
  for (int j = threadIdx.x; j < kTileRows; j += blockDim.x) {
    uint32_t col[4] = {0u, 0u, 0u, 0u};
    for (int i = 0; i < kTileRows; ++i)
      col[i / 32] |= ((s_m[i * 4 + j / 32] >> (j % 32)) & 1u) << (i % 32);
#pragma unroll
    for (int w = 0; w < 4; ++w) mask_t[base + j * 4 + w] = col[w];
  }
}

// Step descriptors of a tile list (order: positions -> tile ids, or null
// for the tiles themselves): (own block, other block, tile id, flags 1 =
// first and 2 = last of the list's run of its own block).
__global__ void k_tile_desc(const int32_t* __restrict__ order, const int32_t* __restrict__ own,
                            const int32_t* __restrict__ oth, int64_t n, int4* __restrict__ desc) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < n; q += stride) {
    const int32_t t = order ? order[q] : int32_t(q);
    const int32_t o = own[t];
    const bool first = q == 0 || own[order ? order[q - 1] : int32_t(q - 1)] != o;
    const bool last = q == n - 1 || own[order ? order[q + 1] : int32_t(q + 1)] != o;
    desc[q] = make_int4(o, oth[t], t, (first ? 1 : 0) | (last ? 2 : 0));
  }
}

// tcol_cb[c] = column block of the c-th column group (its first sorted key)
__global__ void k_group_keys(const int32_t* __restrict__ start, int64_t n_groups,
                             const int32_t* __restrict__ skey, int32_t* __restrict__ blk) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < n_groups; c += stride)
    blk[c] = skey[start[c]];
}

int grid_1d(int64_t n, int num_sms) {
  const int64_t want = (n + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(num_sms) * 8;
  return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

// Stable LSD radix sort of (key, value) pairs, keys in [0, 2^bits) (bit
// patterns of unsigned keys, bits <= 32); the sorted values end in
// *vout_final and the sorted keys in *kout_final (scratch buffers).
gattn_status radix_sort(int32_t* keys, int32_t* vals, int64_t n, int bits, Scratch& scr,
                        cudaStream_t st, int32_t** vout_final, int32_t** kout_final = nullptr) {
  int32_t *kb, *vb, *hist, *offs;
  const int64_t tiles = (n + kTile - 1) / kTile;
  GATTN_CUDA(scr.get(&kb, n));
  GATTN_CUDA(scr.get(&vb, n));
  GATTN_CUDA(scr.get(&hist, tiles * 256));
  GATTN_CUDA(scr.get(&offs, tiles * 256));
  const int passes = (bits + 7) / 8;
  int32_t *kin = keys, *kout = kb, *vin = vals, *vout = vb;
  gattn_status r;
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 8 * pass;
    k_radix_hist<<<(unsigned)tiles, kThreads, 0, st>>>(kin, n, shift, tiles, hist);
    GATTN_CUDA(cudaGetLastError());
    if ((r = exclusive_scan(hist, offs, tiles * 256, scr, st)) != GATTN_OK) return r;
    k_radix_scatter<<<(unsigned)tiles, kThreads, 0, st>>>(kin, vin, kout, vout, n, shift, tiles,
                                                          offs);
    GATTN_CUDA(cudaGetLastError());
    int32_t* t = kin;
    kin = kout;
    kout = t;
    t = vin;
    vin = vout;
    vout = t;
  }
  *vout_final = vin;
  if (kout_final) *kout_final = kin;
  return GATTN_OK;
}

// Transpose of a CSR (row pointer ptr, sources idx, M edges): the column
// pointer ptrT [N+1] and, per CSC position, the CSR edge id (eid [M]) and
// its destination row (dst [M]).  A stable LSD radix sort of the edge ids
// keyed by source keeps every column in CSR edge order.
gattn_status build_csc(const Plan* p, const int32_t* ptr, const int32_t* idx, int64_t M,
                       Scratch& scr, cudaStream_t st, int32_t* ptrT, int32_t* eid, int32_t* dst) {
  const int32_t N = p->N;
  int32_t* counts = nullptr;
  GATTN_CUDA(scr.get(&counts, N + 1));
  GATTN_CUDA(cudaMemsetAsync(counts, 0, (N + 1) * sizeof(int32_t), st));
  if (M) {
    k_count_sources<<<grid_1d(M, p->num_sms), kThreads, 0, st>>>(idx, M, counts);
    GATTN_CUDA(cudaGetLastError());
  }
  gattn_status r;
  if ((r = exclusive_scan(counts, ptrT, N + 1, scr, st)) != GATTN_OK) return r;
  if (M) {
    int32_t *ka, *va, *sorted_eid;
    GATTN_CUDA(scr.get(&ka, M));
    GATTN_CUDA(scr.get(&va, M));
    GATTN_CUDA(cudaMemcpyAsync(ka, idx, M * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    k_iota<<<grid_1d(M, p->num_sms), kThreads, 0, st>>>(va, M);
    GATTN_CUDA(cudaGetLastError());
    int bits = 1;
    while (bits < 31 && (int64_t(1) << bits) < N) ++bits;
    if ((r = radix_sort(ka, va, M, bits, scr, st, &sorted_eid)) != GATTN_OK) return r;
    GATTN_CUDA(cudaMemcpyAsync(eid, sorted_eid, M * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    k_edge_rows<<<grid_1d(M, p->num_sms), kThreads, 0, st>>>(ptr, N, eid, M, dst);
    GATTN_CUDA(cudaGetLastError());
  }
  return GATTN_OK;
}

// The light/heavy split on one side (CSR or CSC): degrees, histogram,
// scans, item list.  Allocates its outputs in the plan.
struct Side {
  int32_t *deg, *hist, *maxdeg, *light_list, *hfirst, *parent;
  int4 *items, *sorted;
  int2* kids;
  int64_t n_light, n_heavy, n_chunks, n_inner;
};

template <typename T>
cudaError_t plan_alloc(Plan* p, T** ptr, size_t n) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, (n ? n : 1) * sizeof(T));
  if (e == cudaSuccess) {
    p->allocs.push_back(q);
    p->device_bytes += (n ? n : 1) * sizeof(T);
  }
  *ptr = reinterpret_cast<T*>(q);
  return e;
}

gattn_status build_side(Plan* p, const int32_t* ptr, Scratch& scr, cudaStream_t st, Side* s) {
  const int32_t N = p->N;
  int32_t *lf, *hf, *nc, *lpos, *hpos, *cpos;
  GATTN_CUDA(plan_alloc(p, &s->deg, N));
  GATTN_CUDA(plan_alloc(p, &s->hist, 33));
  GATTN_CUDA(scr.get(&s->maxdeg, 1));
  GATTN_CUDA(scr.get(&lf, N + 1));
  GATTN_CUDA(scr.get(&hf, N + 1));
  GATTN_CUDA(scr.get(&nc, N + 1));
  GATTN_CUDA(scr.get(&lpos, N + 1));
  GATTN_CUDA(scr.get(&hpos, N + 1));
  GATTN_CUDA(scr.get(&cpos, N + 1));
  GATTN_CUDA(cudaMemsetAsync(s->hist, 0, 33 * sizeof(int32_t), st));
  GATTN_CUDA(cudaMemsetAsync(s->maxdeg, 0, sizeof(int32_t), st));
  k_degrees<<<grid_1d(N + 1, p->num_sms), kThreads, 0, st>>>(ptr, N, p->T, p->C, s->deg, s->hist,
                                                             s->maxdeg, lf, hf, nc);
  GATTN_CUDA(cudaGetLastError());
  gattn_status r;
  if ((r = exclusive_scan(lf, lpos, N + 1, scr, st)) != GATTN_OK) return r;
  if ((r = exclusive_scan(hf, hpos, N + 1, scr, st)) != GATTN_OK) return r;
  if ((r = exclusive_scan(nc, cpos, N + 1, scr, st)) != GATTN_OK) return r;
  int32_t tot[3];
  GATTN_CUDA(cudaMemcpyAsync(&tot[0], lpos + N, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaMemcpyAsync(&tot[1], hpos + N, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaMemcpyAsync(&tot[2], cpos + N, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaStreamSynchronize(st));
  s->n_light = tot[0];
  s->n_heavy = tot[1];
  s->n_chunks = tot[2];
  GATTN_CUDA(plan_alloc(p, &s->light_list, s->n_light));
  GATTN_CUDA(plan_alloc(p, &s->items, s->n_light + s->n_chunks));
  GATTN_CUDA(plan_alloc(p, &s->hfirst, s->n_heavy + 1));
  k_fill_items<<<grid_1d(N, p->num_sms), kThreads, 0, st>>>(ptr, N, p->C, lpos, hpos, cpos,
                                                            s->n_chunks, s->n_heavy, s->light_list,
                                                            s->items, s->hfirst);
  GATTN_CUDA(cudaGetLastError());
  const int64_t n_items = s->n_light + s->n_chunks;
  // merge trees over the heavy nodes' chunks
  {
    int32_t *inner, *ipos;
    GATTN_CUDA(scr.get(&inner, s->n_heavy + 1));
    GATTN_CUDA(scr.get(&ipos, s->n_heavy + 1));
    k_tree_sizes<<<grid_1d(s->n_heavy + 1, p->num_sms), kThreads, 0, st>>>(s->hfirst, s->n_heavy,
                                                                          inner);
    GATTN_CUDA(cudaGetLastError());
    if ((r = exclusive_scan(inner, ipos, s->n_heavy + 1, scr, st)) != GATTN_OK) return r;
    int32_t ni = 0;
    GATTN_CUDA(cudaMemcpyAsync(&ni, ipos + s->n_heavy, 4, cudaMemcpyDeviceToHost, st));
    GATTN_CUDA(cudaStreamSynchronize(st));
    s->n_inner = ni;
    GATTN_CUDA(plan_alloc(p, &s->parent, s->n_chunks + s->n_inner));
    GATTN_CUDA(plan_alloc(p, &s->kids, s->n_inner));
    if (s->n_heavy > 0) {
      k_tree_fill<<<grid_1d(s->n_heavy, p->num_sms), kThreads, 0, st>>>(
          s->hfirst, s->n_heavy, s->n_chunks, ipos, s->parent, s->kids);
      GATTN_CUDA(cudaGetLastError());
    }
  }
  // items by decreasing length (degree binning for the attention kernels)
  GATTN_CUDA(plan_alloc(p, &s->sorted, n_items));
  if (n_items > 0) {
    int32_t *key, *val, *order;
    GATTN_CUDA(scr.get(&key, n_items));
    GATTN_CUDA(scr.get(&val, n_items));
    k_length_keys<<<grid_1d(n_items, p->num_sms), kThreads, 0, st>>>(s->items, n_items, key, val);
    GATTN_CUDA(cudaGetLastError());
    if ((r = radix_sort(key, val, n_items, 9, scr, st, &order)) != GATTN_OK) return r;
    k_gather_sorted<<<grid_1d(n_items, p->num_sms), kThreads, 0, st>>>(s->items, order, n_items,
                                                                       s->sorted);
    GATTN_CUDA(cudaGetLastError());
  }
  return GATTN_OK;
}

// Dense tiles and the residual CSR with its forward split (plan fields
// tile_*, trow_*, *_r).  Needs p->tile_min > 0.
gattn_status tile_build(Plan* p, Scratch& scr, cudaStream_t st) {
  const int32_t N = p->N;
  const int64_t M = p->M;
  const uint32_t nb = uint32_t((int64_t(N) + kTileRows - 1) / kTileRows);
  int32_t *key, *eid, *row, *seid, *skey;
  uint8_t* in_tile;
  GATTN_CUDA(scr.get(&key, M));
  GATTN_CUDA(scr.get(&eid, M));
  GATTN_CUDA(scr.get(&row, M));
  GATTN_CUDA(scr.get(&in_tile, M));
  GATTN_CUDA(cudaMemsetAsync(in_tile, 0, M ? M : 1, st));
  gattn_status r;
  int32_t n_runs = 0, n_tiles = 0;
  int32_t *start = nullptr, *dense = nullptr, *tpos = nullptr;
  if (M) {
    k_block_keys<<<grid_1d(M, p->num_sms), kThreads, 0, st>>>(p->indptr, N, p->indices, M, nb, key,
                                                              eid, row);
    GATTN_CUDA(cudaGetLastError());
    const uint64_t nkeys = uint64_t(nb) * nb;
    int bits = 1;
    while (bits < 32 && (uint64_t(1) << bits) < nkeys) ++bits;
    if ((r = radix_sort(key, eid, M, bits, scr, st, &seid, &skey)) != GATTN_OK) return r;
    int32_t *head, *pos;
    GATTN_CUDA(scr.get(&head, M + 1));
    GATTN_CUDA(scr.get(&pos, M + 1));
    k_run_heads<<<grid_1d(M + 1, p->num_sms), kThreads, 0, st>>>(skey, M, head);
    GATTN_CUDA(cudaGetLastError());
    if ((r = exclusive_scan(head, pos, M + 1, scr, st)) != GATTN_OK) return r;
    GATTN_CUDA(cudaMemcpyAsync(&n_runs, pos + M, 4, cudaMemcpyDeviceToHost, st));
    GATTN_CUDA(cudaStreamSynchronize(st));
    GATTN_CUDA(scr.get(&start, int64_t(n_runs) + 1));
    GATTN_CUDA(scr.get(&dense, int64_t(n_runs) + 1));
    GATTN_CUDA(scr.get(&tpos, int64_t(n_runs) + 1));
    k_run_starts<<<grid_1d(M + 1, p->num_sms), kThreads, 0, st>>>(head, pos, M, start);
    GATTN_CUDA(cudaGetLastError());
    k_run_dense<<<grid_1d(int64_t(n_runs) + 1, p->num_sms), kThreads, 0, st>>>(start, n_runs,
                                                                              p->tile_min, dense);
    GATTN_CUDA(cudaGetLastError());
    if ((r = exclusive_scan(dense, tpos, int64_t(n_runs) + 1, scr, st)) != GATTN_OK) return r;
    GATTN_CUDA(cudaMemcpyAsync(&n_tiles, tpos + n_runs, 4, cudaMemcpyDeviceToHost, st));
    GATTN_CUDA(cudaStreamSynchronize(st));
  }
  p->n_tiles = n_tiles;
  GATTN_CUDA(plan_alloc(p, &p->tile_rb, n_tiles));
  GATTN_CUDA(plan_alloc(p, &p->tile_cb, n_tiles));
  GATTN_CUDA(plan_alloc(p, &p->tile_mask, int64_t(n_tiles) * kTileRows * 4));
  GATTN_CUDA(plan_alloc(p, &p->tile_slot, M));
  GATTN_CUDA(cudaMemsetAsync(p->tile_slot, 0xff, (M ? M : 1) * sizeof(int32_t), st));
  if (n_tiles > 0) {
    int32_t *tbeg, *tend;
    GATTN_CUDA(scr.get(&tbeg, n_tiles));
    GATTN_CUDA(scr.get(&tend, n_tiles));
    k_tile_meta<<<grid_1d(n_runs, p->num_sms), kThreads, 0, st>>>(start, dense, tpos, n_runs, skey,
                                                                 nb, p->tile_rb, p->tile_cb, tbeg,
                                                                 tend);
    GATTN_CUDA(cudaGetLastError());
    k_tile_masks<<<(unsigned)n_tiles, kThreads, 0, st>>>(tbeg, tend, seid, row, p->indices,
                                                        p->tile_mask, in_tile, p->tile_slot);
    GATTN_CUDA(cudaGetLastError());
  }
  // residual CSR
  int32_t* cnt;
  GATTN_CUDA(scr.get(&cnt, int64_t(N) + 1));
  GATTN_CUDA(plan_alloc(p, &p->indptr_r, int64_t(N) + 1));
  const int warp_grid = grid_1d((int64_t(N) + 1) * 32, p->num_sms);
  k_res_count<<<warp_grid, kThreads, 0, st>>>(p->indptr, N, in_tile, cnt);
  GATTN_CUDA(cudaGetLastError());
  if ((r = exclusive_scan(cnt, p->indptr_r, int64_t(N) + 1, scr, st)) != GATTN_OK) return r;
  int32_t mres = 0;
  GATTN_CUDA(cudaMemcpyAsync(&mres, p->indptr_r + N, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaStreamSynchronize(st));
  p->M_res = mres;
  GATTN_CUDA(plan_alloc(p, &p->indices_r, mres));
  GATTN_CUDA(plan_alloc(p, &p->res_eid, mres));
  k_res_fill<<<warp_grid, kThreads, 0, st>>>(p->indptr, N, p->indices, in_tile, p->indptr_r,
                                            p->indices_r, p->res_eid);
  GATTN_CUDA(cudaGetLastError());
  // row blocks with tiles
  int32_t n_trows = 0;
  {
    int32_t *head, *pos;
    GATTN_CUDA(scr.get(&head, int64_t(n_tiles) + 1));
    GATTN_CUDA(scr.get(&pos, int64_t(n_tiles) + 1));
    k_trow_heads<<<grid_1d(int64_t(n_tiles) + 1, p->num_sms), kThreads, 0, st>>>(p->tile_rb,
                                                                                n_tiles, head);
    GATTN_CUDA(cudaGetLastError());
    if ((r = exclusive_scan(head, pos, int64_t(n_tiles) + 1, scr, st)) != GATTN_OK) return r;
    GATTN_CUDA(cudaMemcpyAsync(&n_trows, pos + n_tiles, 4, cudaMemcpyDeviceToHost, st));
    GATTN_CUDA(cudaStreamSynchronize(st));
    p->n_trows = n_trows;
    GATTN_CUDA(plan_alloc(p, &p->trow_rb, n_trows));
    GATTN_CUDA(plan_alloc(p, &p->trow_ptr, int64_t(n_trows) + 1));
    k_trow_fill<<<grid_1d(int64_t(n_tiles) + 1, p->num_sms), kThreads, 0, st>>>(
        p->tile_rb, head, pos, n_tiles, p->trow_rb, p->trow_ptr);
    GATTN_CUDA(cudaGetLastError());
  }
  // forward split of the residual CSR
  Side rs{};
  if ((r = build_side(p, p->indptr_r, scr, st, &rs)) != GATTN_OK) return r;
  p->items_r = rs.items;
  p->sorted_r = rs.sorted;
  p->parent_r = rs.parent;
  p->kids_r = rs.kids;
  p->n_light_r = rs.n_light;
  p->n_chunks_r = rs.n_chunks;
  p->n_inner_r = rs.n_inner;
  GATTN_CUDA(plan_alloc(p, &p->cnt_fwd_r, rs.n_inner));
  GATTN_CUDA(cudaMemsetAsync(p->cnt_fwd_r, 0, (rs.n_inner ? rs.n_inner : 1) * 4, st));
  GATTN_CUDA(plan_alloc(p, &p->cnt_dq_r, rs.n_inner));
  GATTN_CUDA(cudaMemsetAsync(p->cnt_dq_r, 0, (rs.n_inner ? rs.n_inner : 1) * 4, st));
  // residual CSC (backward dK / dV outside the tiles) and its source split
  {
    int32_t* reid;
    GATTN_CUDA(scr.get(&reid, mres));
    GATTN_CUDA(plan_alloc(p, &p->indptrT_r, int64_t(N) + 1));
    GATTN_CUDA(plan_alloc(p, &p->csc_dst_r, mres));
    if ((r = build_csc(p, p->indptr_r, p->indices_r, mres, scr, st, p->indptrT_r, reid,
                       p->csc_dst_r)) != GATTN_OK)
      return r;
    Side ss{};
    if ((r = build_side(p, p->indptrT_r, scr, st, &ss)) != GATTN_OK) return r;
    p->items_src_r = ss.items;
    p->sorted_src_r = ss.sorted;
    p->parent_src_r = ss.parent;
    p->kids_src_r = ss.kids;
    p->n_light_src_r = ss.n_light;
    p->n_chunks_src_r = ss.n_chunks;
    p->n_inner_src_r = ss.n_inner;
    GATTN_CUDA(plan_alloc(p, &p->cnt_dkv_r, ss.n_inner));
    GATTN_CUDA(cudaMemsetAsync(p->cnt_dkv_r, 0, (ss.n_inner ? ss.n_inner : 1) * 4, st));
  }
  // tiles by column block (stable sort of the tile ids by column block, so
  // each column lists its tiles by row block) and the transposed masks
  GATTN_CUDA(plan_alloc(p, &p->tcol_tile, n_tiles));
  GATTN_CUDA(plan_alloc(p, &p->tile_mask_t, int64_t(n_tiles) * kTileRows * 4));
  int32_t n_tcols = 0;
  if (n_tiles > 0) {
    int32_t *ck, *cv, *sid, *skey, *head, *pos, *start;
    GATTN_CUDA(scr.get(&ck, n_tiles));
    GATTN_CUDA(scr.get(&cv, n_tiles));
    GATTN_CUDA(cudaMemcpyAsync(ck, p->tile_cb, n_tiles * sizeof(int32_t),
                               cudaMemcpyDeviceToDevice, st));
    k_iota<<<grid_1d(n_tiles, p->num_sms), kThreads, 0, st>>>(cv, n_tiles);
    GATTN_CUDA(cudaGetLastError());
    int bits = 1;
    while (bits < 31 && (int64_t(1) << bits) < int64_t(nb)) ++bits;
    if ((r = radix_sort(ck, cv, n_tiles, bits, scr, st, &sid, &skey)) != GATTN_OK) return r;
    GATTN_CUDA(cudaMemcpyAsync(p->tcol_tile, sid, n_tiles * sizeof(int32_t),
                               cudaMemcpyDeviceToDevice, st));
    GATTN_CUDA(scr.get(&head, int64_t(n_tiles) + 1));
    GATTN_CUDA(scr.get(&pos, int64_t(n_tiles) + 1));
    k_run_heads<<<grid_1d(int64_t(n_tiles) + 1, p->num_sms), kThreads, 0, st>>>(skey, n_tiles,
                                                                               head);
    GATTN_CUDA(cudaGetLastError());
    if ((r = exclusive_scan(head, pos, int64_t(n_tiles) + 1, scr, st)) != GATTN_OK) return r;
    GATTN_CUDA(cudaMemcpyAsync(&n_tcols, pos + n_tiles, 4, cudaMemcpyDeviceToHost, st));
    GATTN_CUDA(cudaStreamSynchronize(st));
    GATTN_CUDA(plan_alloc(p, &p->tcol_ptr, int64_t(n_tcols) + 1));
    GATTN_CUDA(plan_alloc(p, &p->tcol_cb, n_tcols));
    start = p->tcol_ptr;
    k_run_starts<<<grid_1d(int64_t(n_tiles) + 1, p->num_sms), kThreads, 0, st>>>(head, pos,
                                                                                n_tiles, start);
    GATTN_CUDA(cudaGetLastError());
    k_group_keys<<<grid_1d(n_tcols, p->num_sms), kThreads, 0, st>>>(start, n_tcols, skey,
                                                                    p->tcol_cb);
    GATTN_CUDA(cudaGetLastError());
    k_mask_transpose<<<(unsigned)n_tiles, kTileRows, 0, st>>>(p->tile_mask, p->tile_mask_t);
    GATTN_CUDA(cudaGetLastError());
  }
  GATTN_CUDA(plan_alloc(p, &p->tdesc_row, n_tiles));
  GATTN_CUDA(plan_alloc(p, &p->tdesc_col, n_tiles));
  if (n_tiles > 0) {
    k_tile_desc<<<grid_1d(n_tiles, p->num_sms), kThreads, 0, st>>>(nullptr, p->tile_rb, p->tile_cb,
                                                                   n_tiles, p->tdesc_row);
    GATTN_CUDA(cudaGetLastError());
    k_tile_desc<<<grid_1d(n_tiles, p->num_sms), kThreads, 0, st>>>(p->tcol_tile, p->tile_cb,
                                                                   p->tile_rb, n_tiles, p->tdesc_col);
    GATTN_CUDA(cudaGetLastError());
  } else {
    GATTN_CUDA(plan_alloc(p, &p->tcol_ptr, 1));
    GATTN_CUDA(plan_alloc(p, &p->tcol_cb, 0));
    GATTN_CUDA(cudaMemsetAsync(p->tcol_ptr, 0, sizeof(int32_t), st));
  }
  p->n_tcols = n_tcols;
  return GATTN_OK;
}

}  // namespace

gattn_status plan_build(Plan* p, const int32_t* indptr, const int32_t* indices, cudaStream_t st) {
  const int32_t N = p->N;
  const int64_t M = p->M;
  Scratch scr;
  // 1. validate
  int32_t* err = nullptr;
  GATTN_CUDA(scr.get(&err, 1));
  GATTN_CUDA(cudaMemsetAsync(err, 0, sizeof(int32_t), st));
  k_validate<<<grid_1d(M > N ? M : N + 1, p->num_sms), kThreads, 0, st>>>(indptr, indices, N, M,
                                                                           err);
  GATTN_CUDA(cudaGetLastError());
  int32_t herr = 0;
  GATTN_CUDA(cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaStreamSynchronize(st));
  if (herr) {
    set_error("invalid CSR graph:%s%s%s%s", (herr & 1) ? " indptr[0] != 0;" : "",
              (herr & 2) ? " indptr[N] != M;" : "", (herr & 4) ? " indptr decreases;" : "",
              (herr & 8) ? " source index outside [0, N);" : "");
    return GATTN_ERR_BAD_GRAPH;
  }
  // 2. private copies of the CSR
  GATTN_CUDA(plan_alloc(p, &p->indptr, N + 1));
  GATTN_CUDA(plan_alloc(p, &p->indices, M));
  GATTN_CUDA(cudaMemcpyAsync(p->indptr, indptr, (N + 1) * sizeof(int32_t),
                             cudaMemcpyDeviceToDevice, st));
  if (M) GATTN_CUDA(cudaMemcpyAsync(p->indices, indices, M * sizeof(int32_t),
                                    cudaMemcpyDeviceToDevice, st));
  // 3. destination side
  Side d{};
  gattn_status r = build_side(p, p->indptr, scr, st, &d);
  if (r != GATTN_OK) return r;
  // 4. transpose: out-degrees -> indptrT -> stable sort of edge ids by source
  GATTN_CUDA(plan_alloc(p, &p->indptrT, N + 1));
  GATTN_CUDA(plan_alloc(p, &p->csc_eid, M));
  GATTN_CUDA(plan_alloc(p, &p->csc_dst, M));
  if ((r = build_csc(p, p->indptr, p->indices, M, scr, st, p->indptrT, p->csc_eid, p->csc_dst)) !=
      GATTN_OK)
    return r;
  // 5. source side
  Side s{};
  if ((r = build_side(p, p->indptrT, scr, st, &s)) != GATTN_OK) return r;
  // 6. counters
  GATTN_CUDA(plan_alloc(p, &p->cnt_fwd, d.n_inner));
  GATTN_CUDA(plan_alloc(p, &p->cnt_dq, d.n_inner));
  GATTN_CUDA(plan_alloc(p, &p->cnt_dkv, s.n_inner));
  GATTN_CUDA(plan_alloc(p, &p->cnt_da, 1));
  GATTN_CUDA(plan_alloc(p, &p->err, 1));
  GATTN_CUDA(cudaMemsetAsync(p->err, 0, 4, st));
  GATTN_CUDA(cudaMemsetAsync(p->cnt_fwd, 0, (d.n_inner ? d.n_inner : 1) * 4, st));
  GATTN_CUDA(cudaMemsetAsync(p->cnt_dq, 0, (d.n_inner ? d.n_inner : 1) * 4, st));
  GATTN_CUDA(cudaMemsetAsync(p->cnt_dkv, 0, (s.n_inner ? s.n_inner : 1) * 4, st));
  GATTN_CUDA(cudaMemsetAsync(p->cnt_da, 0, 4, st));
  int32_t mx[2];
  GATTN_CUDA(cudaMemcpyAsync(&mx[0], d.maxdeg, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaMemcpyAsync(&mx[1], s.maxdeg, 4, cudaMemcpyDeviceToHost, st));
  GATTN_CUDA(cudaStreamSynchronize(st));
  p->deg = d.deg;
  p->hist = d.hist;
  p->light = d.light_list;
  p->items = d.items;
  p->hfirst = d.hfirst;
  p->sorted = d.sorted;
  p->parent = d.parent;
  p->kids = d.kids;
  p->n_inner = d.n_inner;
  p->n_light = d.n_light;
  p->n_heavy = d.n_heavy;
  p->n_chunks = d.n_chunks;
  p->outdeg = s.deg;
  p->hist_out = s.hist;
  p->light_src = s.light_list;
  p->items_src = s.items;
  p->hfirst_src = s.hfirst;
  p->sorted_src = s.sorted;
  p->parent_src = s.parent;
  p->kids_src = s.kids;
  p->n_inner_src = s.n_inner;
  p->n_light_src = s.n_light;
  p->n_heavy_src = s.n_heavy;
  p->n_src_chunks = s.n_chunks;
  p->max_deg = mx[0];
  p->max_outdeg = mx[1];
  // 7. dense tiles and the residual CSR
  if (p->tile_min > 0 && (r = tile_build(p, scr, st)) != GATTN_OK) return r;
  return GATTN_OK;
}

}  // namespace gattn
