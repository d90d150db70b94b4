// spmm_api.cu -- C ABI of the weighted SpMM (spmm.cuh, spmm_tile.cu).
#include <algorithm>

#include "attn_launch.cuh"
#include "attn_tile.cuh"
#include "spmm.cuh"
#include "tma.cuh"

namespace gattn {

namespace {

struct SpmmWs {
  size_t part, wperm, tiles, total;
};

size_t up256s(size_t x) { return (x + 255) / 256 * 256; }

bool wsb_ok(const Plan& p, gattn_dtype dt, int64_t F) {
  return p.tile_min > 0 && p.n_tiles > 0 && p.n_tiles * int64_t(kTileRows) * kTileRows < INT32_MAX &&
         dt == GATTN_BF16 && F % 64 == 0;
}

SpmmWs spmm_ws(const Plan& p, gattn_dtype dt, int64_t F) {
  SpmmWs w{};
  const int64_t slots = std::max({p.n_chunks + p.n_inner, p.n_chunks_r + p.n_inner_r,
                                  p.n_src_chunks + p.n_inner_src});
  w.part = 0;
  w.wperm = up256s(size_t(slots) * F * 4);
  w.tiles = up256s(w.wperm + size_t(p.M) * 4);
  w.total = up256s(w.tiles + (wsb_ok(p, dt, F) ? size_t(p.n_tiles) * kTileRows * kTileRows * 2 : 0));
  return w;
}

gattn_status spmm_shape(int32_t F, gattn_dtype dt, int* rb) {
  const int s = dt == GATTN_F32 ? 4 : (dt == GATTN_BF16 ? 2 : 0);
  if (s == 0) {
    set_error("spmm: unknown dtype %d", int(dt));
    return GATTN_ERR_INVALID_ARG;
  }
  const int64_t bytes = int64_t(F) * s;
  if (F <= 0 || (bytes & (bytes - 1)) != 0 || bytes < 32 || bytes > 2048) {
    set_error("spmm: F * sizeof(dtype) must be a power of two in [32, 2048] bytes (F=%d)", F);
    return GATTN_ERR_UNSUPPORTED;
  }
  *rb = int(bytes);
  return GATTN_OK;
}

// weights of the tile edges into their bf16 tile slots
__global__ void k_wsb_scatter(const float* __restrict__ w, const int32_t* __restrict__ slot,
                              int64_t M, __nv_bfloat16* __restrict__ tiles) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < M; e += stride) {
    const int32_t s = slot[e];
    if (s >= 0) tiles[s] = __float2bfloat16_rn(w[e]);
  }
}

// out[k] = w[src[k]]: weights in another edge order (residual CSR, CSC)
__global__ void k_gather_w(const float* __restrict__ w, const int32_t* __restrict__ src, int64_t n,
                           float* __restrict__ out) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < n; k += stride)
    out[k] = w[src[k]];
}

int grid_elems(int64_t n, int sms) {
  return int(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, int64_t(sms) * 16)));
}

#define GATTN_SPMM_CASE(TNAME, RB_) \
  case RB_:                         \
    return launch_spmm_##TNAME##_##RB_(sb, p, sms, st);

gattn_status launch_spmm(gattn_dtype dt, int rb, int sb, const SpmmParams& p, int sms,
                         cudaStream_t st) {
  if (dt == GATTN_F32) {
    switch (rb) { GATTN_FOR_SPMM_ROWS(GATTN_SPMM_CASE, f32) }
  } else {
    switch (rb) { GATTN_FOR_SPMM_ROWS(GATTN_SPMM_CASE, bf16) }
  }
  return GATTN_ERR_UNSUPPORTED;
}
#undef GATTN_SPMM_CASE

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

gattn_status launched(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("gattn_spmm: %s launch failed: %s", what, cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

}  // namespace

}  // namespace gattn

using namespace gattn;

extern "C" {

gattn_status gattn_spmm_workspace_size(const gattn_plan* plan, int32_t F, gattn_dtype dtype,
                                       size_t* bytes) {
  if (!plan || !bytes) {
    set_error("gattn_spmm_workspace_size: plan and bytes must be non-null");
    return GATTN_ERR_INVALID_ARG;
  }
  int rb = 0;
  const gattn_status s = spmm_shape(F, dtype, &rb);
  if (s != GATTN_OK) return s;
  *bytes = spmm_ws(plan->p, dtype, F).total;
  return GATTN_OK;
}

gattn_status gattn_spmm(const gattn_plan* plan, int32_t F, gattn_dtype dtype, const float* w,
                        const void* x, void* y, int32_t transpose, void* workspace,
                        size_t workspace_bytes, gattn_stream_t stream) {
  if (!plan) {
    set_error("gattn_spmm: plan is NULL");
    return GATTN_ERR_INVALID_ARG;
  }
  const Plan& P = plan->p;
  int rb = 0;
  gattn_status s = spmm_shape(F, dtype, &rb);
  if (s != GATTN_OK) return s;
  if (P.N == 0) return GATTN_OK;
  const SpmmWs ws = spmm_ws(P, dtype, F);
  if (!x || !y || x == y || !al16(x) || !al16(y) || (P.M > 0 && (!w || (reinterpret_cast<uintptr_t>(w) & 3))) ||
      !workspace || !al16(workspace) || workspace_bytes < ws.total) {
    set_error("gattn_spmm: x, y need distinct 16-byte aligned device pointers, w a device fp32 "
              "array of M weights, and the workspace %zu bytes (got %zu)", ws.total,
              workspace_bytes);
    return GATTN_ERR_INVALID_ARG;
  }
  char* base = static_cast<char*>(workspace);
  float* part = reinterpret_cast<float*>(base + ws.part);
  float* wperm = reinterpret_cast<float*>(base + ws.wperm);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int es = dtype == GATTN_F32 ? 4 : 2;
  SpmmParams p{};
  if (!encode_rows_map(&p.mx, x, es, dtype == GATTN_BF16, P.N, F)) return GATTN_ERR_CUDA;
  p.N = P.N;
  p.F = F;
  p.y = y;
  p.part = part;
  p.err = P.err;
  const bool wsb = !transpose && wsb_ok(P, dtype, F);
  if (transpose) {  // y = A^T x over the cached CSC, weights in CSC order
    if (P.M) {
      k_gather_w<<<grid_elems(P.M, P.num_sms), 256, 0, st>>>(w, P.csc_eid, P.M, wperm);
      if ((s = launched("weight gather")) != GATTN_OK) return s;
    }
    p.sorted = P.sorted_src;
    p.n_items = P.n_src_chunks + P.n_light_src;
    p.n_chunks = P.n_src_chunks;
    p.idx = P.csc_dst;
    p.w = wperm;
    p.tree = Tree{P.parent_src, P.kids_src, P.n_src_chunks, P.cnt_dkv};
  } else if (wsb) {  // residual edges on the CSR path, then the tiles
    __nv_bfloat16* tiles = reinterpret_cast<__nv_bfloat16*>(base + ws.tiles);
    if (cudaMemsetAsync(tiles, 0, size_t(P.n_tiles) * kTileRows * kTileRows * 2, st) != cudaSuccess) {
      set_error("gattn_spmm: clearing the weight tiles failed");
      return GATTN_ERR_CUDA;
    }
    k_wsb_scatter<<<grid_elems(P.M, P.num_sms), 256, 0, st>>>(w, P.tile_slot, P.M, tiles);
    if ((s = launched("tile weights")) != GATTN_OK) return s;
    if (P.M_res) {
      k_gather_w<<<grid_elems(P.M_res, P.num_sms), 256, 0, st>>>(w, P.res_eid, P.M_res, wperm);
      if ((s = launched("residual weights")) != GATTN_OK) return s;
    }
    p.sorted = P.sorted_r;
    p.n_items = P.n_chunks_r + P.n_light_r;
    p.n_chunks = P.n_chunks_r;
    p.idx = P.indices_r;
    p.w = wperm;
    p.tree = Tree{P.parent_r, P.kids_r, P.n_chunks_r, P.cnt_fwd_r};
  } else {
    p.sorted = P.sorted;
    p.n_items = P.n_chunks + P.n_light;
    p.n_chunks = P.n_chunks;
    p.idx = P.indices;
    p.w = w;
    p.tree = Tree{P.parent, P.kids, P.n_chunks, P.cnt_dq};
  }
  const int64_t edges = transpose ? P.M : (wsb ? P.M_res : P.M);
  if ((s = launch_spmm(dtype, rb, stage_bytes(edges, p.n_items), p, P.num_sms, st)) != GATTN_OK)
    return s;
  if ((s = launched("CSR pass")) != GATTN_OK || !wsb) return s;
  WsbParams t{};
  __nv_bfloat16* tiles = reinterpret_cast<__nv_bfloat16*>(base + ws.tiles);
  if (!encode_tile_map(&t.mw, tiles, P.n_tiles * kTileRows, kTileRows) ||
      !encode_tile_map(&t.mx, x, P.N, F) || !encode_tile_map(&t.my, y, P.N, F))
    return GATTN_ERR_CUDA;
  t.tile_cb = P.tile_cb;
  t.trow_rb = P.trow_rb;
  t.trow_ptr = P.trow_ptr;
  t.n_trows = P.n_trows;
  t.N = P.N;
  t.F = F;
  t.y = y;
  t.err = P.err;
  return launch_wsb_tiles(t, st);
}

}  // extern "C"
