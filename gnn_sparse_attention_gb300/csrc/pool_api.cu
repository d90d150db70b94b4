// pool_api.cu -- C ABI of the max / min pooling layer (pool.cuh).
#include <algorithm>

#include "attn_launch.cuh"
#include "pool.cuh"
#include "tma.cuh"

namespace gattn {

namespace {

struct PoolWs {
  size_t packed, cnt, acc, total;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

PoolWs pool_ws(const Plan& p, int64_t F) {
  PoolWs w{};
  w.packed = 0;
  w.cnt = up256(size_t(p.n_heavy) * F * 8);
  w.acc = up256(w.cnt + size_t(p.n_heavy) * 4);
  w.total = up256(w.acc + size_t(p.N) * F * 4);
  return w;
}

gattn_status pool_shape(int32_t F, gattn_dtype dt, int* rb) {
  const int s = dt == GATTN_F32 ? 4 : (dt == GATTN_BF16 ? 2 : 0);
  if (s == 0) {
    set_error("pooling: unknown dtype %d", int(dt));
    return GATTN_ERR_INVALID_ARG;
  }
  const int64_t bytes = int64_t(F) * s;
  if (F <= 0 || (bytes & (bytes - 1)) != 0 || bytes < 32 || bytes > 2048) {
    set_error("pooling: F * sizeof(dtype) must be a power of two in [32, 2048] bytes (F=%d)", F);
    return GATTN_ERR_UNSUPPORTED;
  }
  *rb = int(bytes);
  return GATTN_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int grid_for_elems(int64_t n, int sms) {
  return int(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, int64_t(sms) * 16)));
}

#define GATTN_POOL_CASE(TNAME, RB_) \
  case RB_:                         \
    return launch_pool_##TNAME##_##RB_(sb, op, p, sms, st);

gattn_status launch_pool(gattn_dtype dt, int rb, int sb, int op, const PoolParams& p, int sms,
                         cudaStream_t st) {
  if (dt == GATTN_F32) {
    switch (rb) { GATTN_FOR_POOL_ROWS(GATTN_POOL_CASE, f32) }
  } else {
    switch (rb) { GATTN_FOR_POOL_ROWS(GATTN_POOL_CASE, bf16) }
  }
  return GATTN_ERR_UNSUPPORTED;
}
#undef GATTN_POOL_CASE

}  // namespace

}  // namespace gattn

using namespace gattn;

extern "C" {

gattn_status gattn_pool_workspace_size(const gattn_plan* plan, int32_t F, gattn_dtype dtype,
                                       size_t* bytes) {
  if (!plan || !bytes) {
    set_error("gattn_pool_workspace_size: plan and bytes must be non-null");
    return GATTN_ERR_INVALID_ARG;
  }
  int rb = 0;
  const gattn_status s = pool_shape(F, dtype, &rb);
  if (s != GATTN_OK) return s;
  *bytes = pool_ws(plan->p, F).total;
  return GATTN_OK;
}

gattn_status gattn_pool_fwd(const gattn_plan* plan, int32_t F, gattn_dtype dtype, int32_t op,
                            const void* x, void* out, int32_t* arg, void* workspace,
                            size_t workspace_bytes, gattn_stream_t stream) {
  if (!plan) {
    set_error("gattn_pool_fwd: plan is NULL");
    return GATTN_ERR_INVALID_ARG;
  }
  const Plan& P = plan->p;
  int rb = 0;
  gattn_status s = pool_shape(F, dtype, &rb);
  if (s != GATTN_OK) return s;
  if (op != GATTN_POOL_MAX && op != GATTN_POOL_MIN) {
    set_error("gattn_pool_fwd: unknown op %d", op);
    return GATTN_ERR_INVALID_ARG;
  }
  if (P.N == 0) return GATTN_OK;
  const PoolWs w = pool_ws(P, F);
  if (!x || !out || !arg || !al16(x) || !al16(out) || !al16(arg) || !workspace ||
      !al16(workspace) || workspace_bytes < w.total) {
    set_error("gattn_pool_fwd: x, out, arg need 16-byte aligned device pointers and the "
              "workspace %zu bytes (got %zu)", w.total, workspace_bytes);
    return GATTN_ERR_INVALID_ARG;
  }
  char* ws = static_cast<char*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (P.n_heavy > 0 && cudaMemsetAsync(ws, 0, w.acc, st) != cudaSuccess) {
    set_error("gattn_pool_fwd: clearing the workspace failed");
    return GATTN_ERR_CUDA;
  }
  PoolParams p{};
  const int es = dtype == GATTN_F32 ? 4 : 2;
  if (!encode_rows_map(&p.mx, x, es, dtype == GATTN_BF16, P.N, F)) return GATTN_ERR_CUDA;
  p.sorted = P.sorted;
  p.items = P.items;
  p.hfirst = P.hfirst;
  p.n_items = P.n_chunks + P.n_light;
  p.n_chunks = P.n_chunks;
  p.N = P.N;
  p.F = F;
  p.idx = P.indices;
  p.out = out;
  p.arg = arg;
  p.packed = reinterpret_cast<unsigned long long*>(ws + w.packed);
  p.cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
  p.err = P.err;
  if ((s = launch_pool(dtype, rb, stage_bytes(P.M, p.n_items), op, p, P.num_sms, st)) != GATTN_OK)
    return s;
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("gattn_pool_fwd: launch failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

gattn_status gattn_pool_bwd(const gattn_plan* plan, int32_t F, gattn_dtype dtype,
                            const int32_t* arg, const void* dout, void* dx, void* workspace,
                            size_t workspace_bytes, gattn_stream_t stream) {
  if (!plan) {
    set_error("gattn_pool_bwd: plan is NULL");
    return GATTN_ERR_INVALID_ARG;
  }
  const Plan& P = plan->p;
  int rb = 0;
  gattn_status s = pool_shape(F, dtype, &rb);
  if (s != GATTN_OK) return s;
  if (P.N == 0) return GATTN_OK;
  const PoolWs w = pool_ws(P, F);
  if (!arg || !dout || !dx || !al16(arg) || !al16(dout) || !al16(dx) || !workspace ||
      !al16(workspace) || workspace_bytes < w.total) {
    set_error("gattn_pool_bwd: arg, dout, dx need 16-byte aligned device pointers and the "
              "workspace %zu bytes (got %zu)", w.total, workspace_bytes);
    return GATTN_ERR_INVALID_ARG;
  }
  float* acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.acc);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t n = int64_t(P.N) * F;
  if (cudaMemsetAsync(acc, 0, size_t(n) * 4, st) != cudaSuccess) {
    set_error("gattn_pool_bwd: clearing the accumulator failed");
    return GATTN_ERR_CUDA;
  }
  const int g4 = grid_for_elems(n / 4, P.num_sms), g1 = grid_for_elems(n, P.num_sms);
  if (dtype == GATTN_F32) {
    pool_bwd_scatter_kernel<float><<<g4, 256, 0, st>>>(arg, static_cast<const float*>(dout), acc,
                                                       n / 4, F);
    pool_bwd_finish_kernel<float><<<g1, 256, 0, st>>>(acc, static_cast<float*>(dx), n);
  } else {
    pool_bwd_scatter_kernel<__nv_bfloat16><<<g4, 256, 0, st>>>(
        arg, static_cast<const __nv_bfloat16*>(dout), acc, n / 4, F);
    pool_bwd_finish_kernel<__nv_bfloat16><<<g1, 256, 0, st>>>(acc, static_cast<__nv_bfloat16*>(dx),
                                                             n);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("gattn_pool_bwd: launch failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

}  // extern "C"
