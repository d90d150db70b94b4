// reorder.cu -- node relabelling for gather locality (host) and the row
// permutation of dense tensors (device).
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology" and results: graph reordering, which
// the pages find helps neighbour-parallel (gather-dominated) kernels on
// high-degree graphs and barely matters on low-degree ones.  The pages name
// no method; two textbook relabellings are offered:
//   degree : nodes by decreasing total degree (in + out), ties by id -- the
//            most-gathered rows end up next to each other;
//   RCM    : reverse Cuthill-McKee on the undirected simple graph, roots of
//            least (degree, id), neighbours visited in (degree, id) order --
//            neighbours get nearby ids, which narrows the gather footprint.
// A relabelling is a one-off host preprocessing step; the permutation of
// the feature rows (and back) runs on the device.
#include <algorithm>
#include <numeric>
#include <vector>

#include "gattn_internal.cuh"

namespace gattn {

namespace {

bool is_permutation(const int32_t* perm, int32_t N) {
  std::vector<uint8_t> hit(size_t(N), 0);
  for (int32_t i = 0; i < N; ++i) {
    const int32_t v = perm[i];
    if (v < 0 || v >= N || hit[size_t(v)]) return false;
    hit[size_t(v)] = 1;
  }
  return true;
}

bool valid_csr(const int32_t* ptr, const int32_t* idx, int32_t N, int64_t M) {
  if (ptr[0] != 0 || ptr[N] != M) return false;
  for (int32_t i = 0; i < N; ++i)
    if (ptr[i + 1] < ptr[i]) return false;
  for (int64_t e = 0; e < M; ++e)
    if (idx[e] < 0 || idx[e] >= N) return false;
  return true;
}

void degree_order(const int32_t* ptr, const int32_t* idx, int32_t N, int64_t M, int32_t* perm) {
  std::vector<int64_t> deg(size_t(N), 0);
  for (int32_t i = 0; i < N; ++i) deg[size_t(i)] += ptr[i + 1] - ptr[i];
  for (int64_t e = 0; e < M; ++e) deg[size_t(idx[e])] += 1;
  std::iota(perm, perm + N, 0);
  std::stable_sort(perm, perm + N, [&](int32_t a, int32_t b) { return deg[size_t(a)] > deg[size_t(b)]; });
}

void rcm_order(const int32_t* ptr, const int32_t* idx, int32_t N, int64_t M, int32_t* perm) {
  // undirected simple graph in CSR form: both directions of every non-loop
  // edge, each list sorted and deduplicated
  std::vector<int64_t> off(size_t(N) + 1, 0);
  for (int32_t i = 0; i < N; ++i)
    for (int64_t e = ptr[i]; e < ptr[i + 1]; ++e)
      if (idx[e] != i) {
        ++off[size_t(i) + 1];
        ++off[size_t(idx[e]) + 1];
      }
  std::partial_sum(off.begin(), off.end(), off.begin());
  std::vector<int32_t> nbr(static_cast<size_t>(off[size_t(N)]));
  {
    std::vector<int64_t> pos(off.begin(), off.end() - 1);
    for (int32_t i = 0; i < N; ++i)
      for (int64_t e = ptr[i]; e < ptr[i + 1]; ++e) {
        const int32_t j = idx[e];
        if (j == i) continue;
        nbr[size_t(pos[size_t(i)]++)] = j;
        nbr[size_t(pos[size_t(j)]++)] = i;
      }
  }
  std::vector<int64_t> len(static_cast<size_t>(N));
  for (int32_t i = 0; i < N; ++i) {
    auto b = nbr.begin() + off[size_t(i)], e = nbr.begin() + off[size_t(i) + 1];
    std::sort(b, e);
    len[size_t(i)] = std::unique(b, e) - b;
  }
  auto before = [&](int32_t a, int32_t b) {
    return len[size_t(a)] != len[size_t(b)] ? len[size_t(a)] < len[size_t(b)] : a < b;
  };
  std::vector<int32_t> roots(static_cast<size_t>(N));
  std::iota(roots.begin(), roots.end(), 0);
  std::sort(roots.begin(), roots.end(), before);
  std::vector<uint8_t> seen(size_t(N), 0);
  std::vector<int32_t> order;
  order.reserve(size_t(N));
  std::vector<int32_t> fresh;
  size_t head = 0, next_root = 0;
  while (order.size() < size_t(N)) {
    while (seen[size_t(roots[next_root])]) ++next_root;
    const int32_t r = roots[next_root];
    seen[size_t(r)] = 1;
    order.push_back(r);
    while (head < order.size()) {
      const int32_t v = order[head++];
      fresh.clear();
      for (int64_t k = off[size_t(v)]; k < off[size_t(v)] + len[size_t(v)]; ++k)
        if (!seen[size_t(nbr[size_t(k)])]) fresh.push_back(nbr[size_t(k)]);
      std::sort(fresh.begin(), fresh.end(), before);
      for (int32_t w : fresh) {
        seen[size_t(w)] = 1;
        order.push_back(w);
      }
    }
  }
  std::reverse_copy(order.begin(), order.end(), perm);
}

// dst row i <- src row perm[i] (gather) or dst row perm[i] <- src row i
// (scatter); one warp per row, 16-byte pieces.  Indices outside [0, N) are
// skipped.
__global__ void k_permute_rows(const uint4* __restrict__ src, uint4* __restrict__ dst,
                               const int32_t* __restrict__ perm, int32_t N, int64_t pieces,
                               int scatter) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < N; i += warps) {
    const int32_t p = perm[i];
    if (p < 0 || p >= N) continue;
    const int64_t s = scatter ? i : p, d = scatter ? p : i;
    for (int64_t c = lane; c < pieces; c += 32) dst[d * pieces + c] = src[s * pieces + c];
  }
}

}  // namespace

}  // namespace gattn

using namespace gattn;

extern "C" {

gattn_status gattn_reorder(const int32_t* indptr, const int32_t* indices, int32_t N, int64_t M,
                           int32_t kind, int32_t* perm) {
  if (N < 0 || M < 0 || !indptr || (M > 0 && !indices) || (N > 0 && !perm)) {
    set_error("gattn_reorder: bad sizes or null host pointers");
    return GATTN_ERR_INVALID_ARG;
  }
  if (kind != GATTN_REORDER_DEGREE && kind != GATTN_REORDER_RCM) {
    set_error("gattn_reorder: unknown relabelling kind %d", kind);
    return GATTN_ERR_INVALID_ARG;
  }
  if (!valid_csr(indptr, indices, N, M)) {
    set_error("gattn_reorder: invalid CSR graph");
    return GATTN_ERR_BAD_GRAPH;
  }
  try {
    if (kind == GATTN_REORDER_DEGREE) degree_order(indptr, indices, N, M, perm);
    else rcm_order(indptr, indices, N, M, perm);
  } catch (const std::bad_alloc&) {
    set_error("gattn_reorder: host allocation failed");
    return GATTN_ERR_OOM;
  }
  return GATTN_OK;
}

gattn_status gattn_permute_csr(const int32_t* indptr, const int32_t* indices, int32_t N,
                               int64_t M, const int32_t* perm, int32_t* indptr_out,
                               int32_t* indices_out) {
  if (N < 0 || M < 0 || !indptr || !indptr_out || (M > 0 && (!indices || !indices_out)) ||
      (N > 0 && !perm)) {
    set_error("gattn_permute_csr: bad sizes or null host pointers");
    return GATTN_ERR_INVALID_ARG;
  }
  if (!valid_csr(indptr, indices, N, M)) {
    set_error("gattn_permute_csr: invalid CSR graph");
    return GATTN_ERR_BAD_GRAPH;
  }
  if (!is_permutation(perm, N)) {
    set_error("gattn_permute_csr: perm is not a permutation of [0, N)");
    return GATTN_ERR_INVALID_ARG;
  }
  try {
    std::vector<int32_t> inv(static_cast<size_t>(N));
    for (int32_t i = 0; i < N; ++i) inv[size_t(perm[i])] = i;
    indptr_out[0] = 0;
    int64_t o = 0;
    for (int32_t i = 0; i < N; ++i) {
      const int32_t old = perm[i];
      const int64_t first = o;
      for (int64_t e = indptr[old]; e < indptr[old + 1]; ++e) indices_out[o++] = inv[size_t(indices[e])];
      std::sort(indices_out + first, indices_out + o);
      indptr_out[i + 1] = int32_t(o);
    }
  } catch (const std::bad_alloc&) {
    set_error("gattn_permute_csr: host allocation failed");
    return GATTN_ERR_OOM;
  }
  return GATTN_OK;
}

gattn_status gattn_permute_rows(const void* src, void* dst, const int32_t* perm, int32_t N,
                                int64_t row_bytes, int32_t inverse, gattn_stream_t stream) {
  if (N < 0 || row_bytes <= 0 || row_bytes % 16 != 0) {
    set_error("gattn_permute_rows: need N >= 0 and row_bytes a positive multiple of 16");
    return GATTN_ERR_INVALID_ARG;
  }
  if (N == 0) return GATTN_OK;
  if (!src || !dst || !perm || src == dst || (reinterpret_cast<uintptr_t>(src) & 15) ||
      (reinterpret_cast<uintptr_t>(dst) & 15)) {
    set_error("gattn_permute_rows: src and dst must be distinct 16-byte aligned device pointers");
    return GATTN_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    set_error("gattn_permute_rows: no CUDA device");
    return GATTN_ERR_CUDA;
  }
  const int64_t want = (int64_t(N) * 32 + kThreads - 1) / kThreads;
  const int grid = int(std::min<int64_t>(want, int64_t(sms) * 16));
  k_permute_rows<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), perm, N, row_bytes / 16,
      inverse ? 1 : 0);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("gattn_permute_rows: launch failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

}  // extern "C"
