// api.cu -- the C ABI (include/gattn.h): argument checks, workspace layout,
// plan lifetime and the launch sequence of the forward and backward passes.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "attn_launch.cuh"
#include "attn_tile.cuh"
#include "tma.cuh"

namespace gattn {

namespace {
thread_local char g_err[512] = "";
}

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

gattn_status plan_build(Plan* p, const int32_t* indptr, const int32_t* indices, cudaStream_t st);

namespace {

size_t dtype_size(gattn_dtype dt) { return dt == GATTN_F32 ? 4 : (dt == GATTN_BF16 ? 2 : 0); }
bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

gattn_status check_shape(int32_t H, int32_t D, gattn_dtype dt, int* rb) {
  const size_t s = dtype_size(dt);
  if (s == 0) {
    set_error("unknown dtype %d", (int)dt);
    return GATTN_ERR_INVALID_ARG;
  }
  if (H <= 0 || D <= 0) {
    set_error("H and D must be positive (H=%d, D=%d)", H, D);
    return GATTN_ERR_INVALID_ARG;
  }
  const int64_t dbytes = int64_t(D) * s, row = int64_t(H) * dbytes;
  if (!pow2(H) || !pow2(D) || dbytes < 16 || dbytes > 512 || row < 32 || row > 2048) {
    set_error("unsupported head layout H=%d D=%d dtype=%s: need powers of two with "
              "16 <= D*size <= 512 and 32 <= H*D*size <= 2048 bytes",
              H, D, dt == GATTN_F32 ? "f32" : "bf16");
    return GATTN_ERR_UNSUPPORTED;
  }
  *rb = (int)row;
  return GATTN_OK;
}

struct Workspace {
  size_t fwd_part, dq_part, delta, dkv_part, da_part, total;
  int pstride;
};

Workspace ws_layout(const Plan& p, int H, int D) {
  Workspace w{};
  const size_t HD = size_t(H) * D;
  w.pstride = (int)align_up(HD + 2 * size_t(H), 4);
  size_t off = 0;
  w.fwd_part = off;
  const size_t slots = size_t(p.n_chunks + p.n_inner);
  const size_t slots_res = size_t(p.n_chunks_r + p.n_inner_r);  // residual forward (tiles)
  const size_t slots_src_full = size_t(p.n_src_chunks + p.n_inner_src);
  const size_t slots_src_res = size_t(p.n_chunks_src_r + p.n_inner_src_r);
  const size_t slots_src = slots_src_full > slots_src_res ? slots_src_full : slots_src_res;
  off = align_up(off + (slots > slots_res ? slots : slots_res) * w.pstride * 4, 256);
  w.dq_part = off;
  off = align_up(off + (slots > slots_res ? slots : slots_res) * HD * 4, 256);
  w.delta = off;
  off = align_up(off + size_t(p.N) * 2 * H * 4, 256);  // (lse log2(e), Delta) per node
  w.dkv_part = off;
  off = align_up(off + slots_src * 2 * HD * 4, 256);
  w.da_part = off;
  off = align_up(off + size_t(p.num_sms) * kMaxBlocksPerSm * HD * 4, 256);
  w.total = off;
  return w;
}

gattn_status check_score(const gattn_score* sc, int32_t D, float* qmul, float* scale,
                         float* slope) {
  if (!sc) {
    set_error("score is NULL");
    return GATTN_ERR_INVALID_ARG;
  }
  if (sc->kind == GATTN_SCORE_DOT) {
    *scale = sc->scale != 0.f ? sc->scale : (float)(1.0 / std::sqrt((double)D));
    *qmul = *scale * kLog2e;
    *slope = 0.f;
    return GATTN_OK;
  }
  if (sc->kind == GATTN_SCORE_GATV2) {
    if (!sc->a || !aligned(sc->a, 4)) {
      set_error("GATv2 score needs a device pointer a[H*D] (4-byte aligned)");
      return GATTN_ERR_INVALID_ARG;
    }
    *scale = 1.f;
    *qmul = 1.f;
    *slope = sc->neg_slope;
    return GATTN_OK;
  }
  set_error("unknown score kind %d", sc->kind);
  return GATTN_ERR_INVALID_ARG;
}

gattn_status check_tensor(const void* t, const char* name) {
  if (!t || !aligned(t, 16)) {
    set_error("%s must be a non-null 16-byte aligned device pointer", name);
    return GATTN_ERR_INVALID_ARG;
  }
  return GATTN_OK;
}

// A tiled plan runs its dense tiles on the tensor cores for bf16 I/O, the
// dot score and D = 64 or 128; other layouts take the CSR path over every
// edge.
bool tile_path(const Plan& p, gattn_dtype dt, int kind, int D) {
  return p.tile_min > 0 && p.n_tiles > 0 && dt == GATTN_BF16 && kind == GATTN_SCORE_DOT &&
         (D == 64 || D == 128);
}

gattn_status launched(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s launch failed: %s", what, cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

}  // namespace

// switch key of a (row bytes, stage bytes) pair
#define GATTN_STAGE_KEY(RB_, SB_) ((RB_) * 16 + ((SB_) == kStageSmall ? 1 : 2))
#define GATTN_ROW_CASE(PASS_NAME, PT, TNAME, RB_, SB_) \
  case GATTN_STAGE_KEY(RB_, SB_):                      \
    return launch_##PASS_NAME##_##TNAME##_##RB_##_##SB_(db, kind, p, num_sms, st, g);

gattn_status launch_fwd(gattn_dtype dt, int rb, int db, int kind, int sb, const FwdParams& p,
                        int num_sms, cudaStream_t st, int* g) {
  if (dt == GATTN_F32) {
    switch (GATTN_STAGE_KEY(rb, sb)) { GATTN_FOR_ROWS(GATTN_ROW_CASE, fwd, FwdParams, f32) }
  } else {
    switch (GATTN_STAGE_KEY(rb, sb)) { GATTN_FOR_ROWS(GATTN_ROW_CASE, fwd, FwdParams, bf16) }
  }
  return GATTN_ERR_UNSUPPORTED;
}
gattn_status launch_bwd_csr(gattn_dtype dt, int rb, int db, int kind, int sb, const BwdParams& p,
                            int num_sms, cudaStream_t st, int* g) {
  if (dt == GATTN_F32) {
    switch (GATTN_STAGE_KEY(rb, sb)) { GATTN_FOR_ROWS(GATTN_ROW_CASE, csr, BwdParams, f32) }
  } else {
    switch (GATTN_STAGE_KEY(rb, sb)) { GATTN_FOR_ROWS(GATTN_ROW_CASE, csr, BwdParams, bf16) }
  }
  return GATTN_ERR_UNSUPPORTED;
}
gattn_status launch_bwd_csc(gattn_dtype dt, int rb, int db, int kind, int sb, const BwdParams& p,
                            int num_sms, cudaStream_t st, int* g) {
  if (dt == GATTN_F32) {
    switch (GATTN_STAGE_KEY(rb, sb)) { GATTN_FOR_ROWS(GATTN_ROW_CASE, csc, BwdParams, f32) }
  } else {
    switch (GATTN_STAGE_KEY(rb, sb)) { GATTN_FOR_ROWS(GATTN_ROW_CASE, csc, BwdParams, bf16) }
  }
  return GATTN_ERR_UNSUPPORTED;
}
#undef GATTN_ROW_CASE
#undef GATTN_STAGE_KEY

}  // namespace gattn

using namespace gattn;

#define GATTN_REQUIRE(cond, code, ...) \
  do {                                 \
    if (!(cond)) {                     \
      set_error(__VA_ARGS__);          \
      return code;                     \
    }                                  \
  } while (0)

extern "C" {

const char* gattn_last_error(void) { return g_err; }

const char* gattn_version(void) { return "gattn 0.1.0 sm_103a"; }

gattn_status gattn_plan_create(const int32_t* indptr, const int32_t* indices, int32_t N,
                               int64_t M, const gattn_plan_opts* opts, gattn_stream_t stream,
                               gattn_plan** out) {
  g_err[0] = 0;
  GATTN_REQUIRE(out != nullptr, GATTN_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  GATTN_REQUIRE(N >= 0 && M >= 0 && M < (int64_t(1) << 31), GATTN_ERR_INVALID_ARG,
                "need N >= 0 and 0 <= M < 2^31 (N=%d, M=%lld)", N, (long long)M);
  GATTN_REQUIRE(indptr != nullptr && (M == 0 || indices != nullptr), GATTN_ERR_INVALID_ARG,
                "indptr/indices must be device pointers");
  // Default threshold and chunk: the largest work item should stay small
  // next to one warp's share of the edges (about M / (256 * SMs) edges per
  // item keeps the longest-first schedule balanced), between 32 and 256.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    set_error("no CUDA device: %s", cudaGetErrorString(cudaGetLastError()));
    return GATTN_ERR_CUDA;
  }
  int T = 32;
  while (T < kMaxItemEdges && int64_t(2 * T) * 256 * sms <= M) T *= 2;
  int C = T;
  if (opts) {
    if (opts->heavy_threshold > 0) T = opts->heavy_threshold;
    if (opts->chunk > 0) C = opts->chunk;
    GATTN_REQUIRE(T <= kMaxItemEdges && C <= kMaxItemEdges, GATTN_ERR_INVALID_ARG,
                  "heavy_threshold and chunk must be at most %d (got %d, %d)", kMaxItemEdges, T,
                  C);
  }
  int32_t tile_min = 0;
  if (opts && opts->tile_enable) {
    GATTN_REQUIRE(N <= (1 << 23), GATTN_ERR_UNSUPPORTED,
                  "the dense-tile split needs N <= 2^23 (got %d)", N);
    const float dens = opts->tile_density > 0.f ? opts->tile_density : 0.0625f;
    GATTN_REQUIRE(dens <= 1.f, GATTN_ERR_INVALID_ARG, "tile_density must be at most 1 (got %g)",
                  (double)dens);
    const double need = std::ceil(double(dens) * kTileRows * kTileRows);
    tile_min = need < 1.0 ? 1 : int32_t(need);
  }
  gattn_plan* h = new (std::nothrow) gattn_plan();
  GATTN_REQUIRE(h != nullptr, GATTN_ERR_OOM, "host allocation failed");
  Plan& p = h->p;
  p.N = N;
  p.M = M;
  p.T = T;
  p.C = C;
  p.device = dev;
  p.num_sms = sms;
  p.tile_min = tile_min;
  const gattn_status s = plan_build(&p, indptr, indices, reinterpret_cast<cudaStream_t>(stream));
  if (s != GATTN_OK) {
    for (void* q : p.allocs) cudaFree(q);
    delete h;
    return s;
  }
  *out = h;
  return GATTN_OK;
}

gattn_status gattn_plan_destroy(gattn_plan* plan) {
  if (!plan) return GATTN_OK;
  cudaError_t e = cudaSuccess;
  for (void* q : plan->p.allocs) {
    const cudaError_t r = cudaFree(q);
    if (r != cudaSuccess) e = r;
  }
  delete plan;
  if (e != cudaSuccess) {
    set_error("cudaFree failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

gattn_status gattn_plan_get_info(const gattn_plan* plan, gattn_plan_info* info) {
  GATTN_REQUIRE(plan && info, GATTN_ERR_INVALID_ARG, "plan and info must be non-null");
  const Plan& p = plan->p;
  info->N = p.N;
  info->M = p.M;
  info->heavy_threshold = p.T;
  info->chunk = p.C;
  info->n_light = p.n_light;
  info->n_heavy = p.n_heavy;
  info->n_chunks = p.n_chunks;
  info->n_light_src = p.n_light_src;
  info->n_heavy_src = p.n_heavy_src;
  info->n_src_chunks = p.n_src_chunks;
  info->max_deg = p.max_deg;
  info->max_outdeg = p.max_outdeg;
  info->device_bytes = p.device_bytes;
  info->n_tiles = p.n_tiles;
  info->n_tile_rows = p.n_trows;
  info->tile_edges = p.tile_min > 0 ? p.M - p.M_res : 0;
  info->tile_min_edges = p.tile_min;
  return GATTN_OK;
}

static gattn_status copy_out(int32_t* host, const void* dev, size_t n) {
  if (!host || n == 0) return GATTN_OK;
  const cudaError_t e = cudaMemcpy(host, dev, n * sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_error("cudaMemcpy failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}

static gattn_status copy_chunks(int32_t* host, const int4* items, int64_t n) {
  if (!host || n == 0) return GATTN_OK;
  int4* tmp = new (std::nothrow) int4[n];
  GATTN_REQUIRE(tmp != nullptr, GATTN_ERR_OOM, "host allocation failed");
  const cudaError_t e = cudaMemcpy(tmp, items, n * sizeof(int4), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    delete[] tmp;
    set_error("cudaMemcpy failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  for (int64_t c = 0; c < n; ++c) {
    host[3 * c] = tmp[c].x;
    host[3 * c + 1] = tmp[c].y;
    host[3 * c + 2] = tmp[c].z;
  }
  delete[] tmp;
  return GATTN_OK;
}

gattn_status gattn_plan_export(const gattn_plan* plan, int32_t* deg, int32_t* hist,
                               int32_t* light, int32_t* chunks, int32_t* indptrT,
                               int32_t* csc_dst, int32_t* csc_eid, int32_t* outdeg,
                               int32_t* hist_out, int32_t* light_src, int32_t* src_chunks) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = plan->p;
  gattn_status s;
  if ((s = copy_out(deg, p.deg, p.N)) != GATTN_OK) return s;
  if ((s = copy_out(hist, p.hist, 33)) != GATTN_OK) return s;
  if ((s = copy_out(light, p.light, p.n_light)) != GATTN_OK) return s;
  if ((s = copy_chunks(chunks, p.items, p.n_chunks)) != GATTN_OK) return s;
  if ((s = copy_out(indptrT, p.indptrT, size_t(p.N) + 1)) != GATTN_OK) return s;
  if ((s = copy_out(csc_dst, p.csc_dst, p.M)) != GATTN_OK) return s;
  if ((s = copy_out(csc_eid, p.csc_eid, p.M)) != GATTN_OK) return s;
  if ((s = copy_out(outdeg, p.outdeg, p.N)) != GATTN_OK) return s;
  if ((s = copy_out(hist_out, p.hist_out, 33)) != GATTN_OK) return s;
  if ((s = copy_out(light_src, p.light_src, p.n_light_src)) != GATTN_OK) return s;
  if ((s = copy_chunks(src_chunks, p.items_src, p.n_src_chunks)) != GATTN_OK) return s;
  return GATTN_OK;
}

gattn_status gattn_plan_export_tiles(const gattn_plan* plan, int32_t* tile_rb, int32_t* tile_cb,
                                     uint32_t* masks, int32_t* indptr_r, int32_t* indices_r) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = plan->p;
  GATTN_REQUIRE(p.tile_min > 0, GATTN_ERR_INVALID_ARG, "the plan was built without tile_enable");
  gattn_status s;
  if ((s = copy_out(tile_rb, p.tile_rb, p.n_tiles)) != GATTN_OK) return s;
  if ((s = copy_out(tile_cb, p.tile_cb, p.n_tiles)) != GATTN_OK) return s;
  if ((s = copy_out(reinterpret_cast<int32_t*>(masks), p.tile_mask,
                    size_t(p.n_tiles) * kTileRows * 4)) != GATTN_OK)
    return s;
  if ((s = copy_out(indptr_r, p.indptr_r, size_t(p.N) + 1)) != GATTN_OK) return s;
  if ((s = copy_out(indices_r, p.indices_r, p.M_res)) != GATTN_OK) return s;
  return GATTN_OK;
}

gattn_status gattn_plan_export_tile_bwd(const gattn_plan* plan, int64_t* n_tcols,
                                        int32_t* tcol_cb, int32_t* tcol_ptr, int32_t* tcol_tile,
                                        uint32_t* masks_t, int32_t* indptrT_r,
                                        int32_t* csc_dst_r) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = plan->p;
  GATTN_REQUIRE(p.tile_min > 0, GATTN_ERR_INVALID_ARG, "the plan was built without tile_enable");
  if (n_tcols) *n_tcols = p.n_tcols;
  gattn_status s;
  if ((s = copy_out(tcol_cb, p.tcol_cb, p.n_tcols)) != GATTN_OK) return s;
  if ((s = copy_out(tcol_ptr, p.tcol_ptr, size_t(p.n_tcols) + 1)) != GATTN_OK) return s;
  if ((s = copy_out(tcol_tile, p.tcol_tile, p.n_tiles)) != GATTN_OK) return s;
  if ((s = copy_out(reinterpret_cast<int32_t*>(masks_t), p.tile_mask_t,
                    size_t(p.n_tiles) * kTileRows * 4)) != GATTN_OK)
    return s;
  if ((s = copy_out(indptrT_r, p.indptrT_r, size_t(p.N) + 1)) != GATTN_OK) return s;
  if ((s = copy_out(csc_dst_r, p.csc_dst_r, p.M_res)) != GATTN_OK) return s;
  return GATTN_OK;
}

gattn_status gattn_plan_check_errors(const gattn_plan* plan) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = plan->p;
  cudaError_t e = cudaDeviceSynchronize();
  int32_t flag = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&flag, p.err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_error("checking the plan's error flag failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  if (flag) {
    // A warp that gave up left its items unfinished, so an arrival counter
    // of a merge tree may hold a count of chunks that never completed: clear
    // every counter (the device is idle) so that the next call starts clean.
    struct {
      int32_t* c;
      int64_t n;
    } cnt[] = {{p.cnt_fwd, p.n_inner},       {p.cnt_dq, p.n_inner},
               {p.cnt_dkv, p.n_inner_src},   {p.cnt_da, 1},
               {p.cnt_fwd_r, p.n_inner_r},   {p.cnt_dq_r, p.n_inner_r},
               {p.cnt_dkv_r, p.n_inner_src_r}, {p.err, 1}};
    for (const auto& x : cnt)
      if (x.c && e == cudaSuccess) e = cudaMemset(x.c, 0, size_t(x.n > 0 ? x.n : 1) * 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      set_error("clearing the plan's counters failed: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    set_error("a kernel gave up waiting for its asynchronous copies");
    return GATTN_ERR_TIMEOUT;
  }
  return GATTN_OK;
}

gattn_status gattn_plan_set_wait_test(gattn_plan* plan, int32_t fail_first_wait) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  plan->p.fail_first_wait = fail_first_wait != 0;
  return GATTN_OK;
}

gattn_status gattn_workspace_size(const gattn_plan* plan, int32_t H, int32_t D,
                                  gattn_dtype dtype, size_t* bytes) {
  GATTN_REQUIRE(plan && bytes, GATTN_ERR_INVALID_ARG, "plan and bytes must be non-null");
  int rb = 0;
  const gattn_status s = check_shape(H, D, dtype, &rb);
  if (s != GATTN_OK) return s;
  *bytes = ws_layout(plan->p, H, D).total;
  return GATTN_OK;
}

gattn_status gattn_fwd(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                       const void* Q, const void* K, const void* V, const gattn_score* score,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       gattn_stream_t stream) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = plan->p;
  int rb = 0;
  gattn_status s = check_shape(H, D, dtype, &rb);
  if (s != GATTN_OK) return s;
  FwdParams f{};
  float scale = 1.f;
  if ((s = check_score(score, D, &f.qmul, &scale, &f.slope)) != GATTN_OK) return s;
  if (p.N == 0) return GATTN_OK;
  if ((s = check_tensor(Q, "Q")) || (s = check_tensor(K, "K")) || (s = check_tensor(V, "V")) ||
      (s = check_tensor(out, "out")))
    return s;
  GATTN_REQUIRE(lse && aligned(lse, 4), GATTN_ERR_INVALID_ARG, "lse must be a device pointer");
  const Workspace w = ws_layout(p, H, D);
  GATTN_REQUIRE(workspace && aligned(workspace, 16) && workspace_bytes >= w.total,
                GATTN_ERR_INVALID_ARG, "workspace needs %zu bytes (16-byte aligned), got %zu",
                w.total, workspace_bytes);
  char* ws = static_cast<char*>(workspace);
  // dense tiles on the tensor cores: the CSR pass covers the residual edges
  const bool tiles = tile_path(p, dtype, score->kind, D);
  f.items = tiles ? p.items_r : p.items;
  f.sorted = tiles ? p.sorted_r : p.sorted;
  f.n_items = tiles ? p.n_chunks_r + p.n_light_r : p.n_chunks + p.n_light;
  f.n_chunks = tiles ? p.n_chunks_r : p.n_chunks;
  f.N = p.N;
  {
    const int es = (int)dtype_size(dtype);
    const bool bf = dtype == GATTN_BF16;
    const int64_t HD = int64_t(H) * D;
    if (!encode_rows_map(&f.mq, Q, es, bf, p.N, HD) || !encode_rows_map(&f.mk, K, es, bf, p.N, HD) ||
        !encode_rows_map(&f.mv, V, es, bf, p.N, HD))
      return GATTN_ERR_CUDA;
  }
  f.indices = tiles ? p.indices_r : p.indices;
  f.Q = Q;
  f.K = K;
  f.V = V;
  f.out = out;
  f.lse = lse;
  f.a = score->a;
  f.H = H;
  f.D = D;
  f.part = reinterpret_cast<float*>(ws + w.fwd_part);
  f.pstride = w.pstride;
  f.tree = tiles ? Tree{p.parent_r, p.kids_r, p.n_chunks_r, p.cnt_fwd_r}
                 : Tree{p.parent, p.kids, p.n_chunks, p.cnt_fwd};
  f.err = p.err;
  f.fail_first_wait = p.fail_first_wait;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int sb = tiles ? stage_bytes(p.M_res, p.n_chunks_r + p.n_light_r)
                       : stage_bytes(p.M, p.n_chunks + p.n_light);
  if ((s = launch_fwd(dtype, rb, D * (int)dtype_size(dtype), score->kind, sb, f, p.num_sms, st,
                      nullptr)) != GATTN_OK)
    return s;
  if ((s = launched("forward")) != GATTN_OK || !tiles) return s;
  TileParams tp{};
  const int64_t HD = int64_t(H) * D;
  if (!encode_tile_map(&tp.mq, Q, p.N, HD) || !encode_tile_map(&tp.mk, K, p.N, HD) ||
      !encode_tile_map(&tp.mv, V, p.N, HD) || !encode_tile_map(&tp.mo, out, p.N, HD))
    return GATTN_ERR_CUDA;
  tp.mask = p.tile_mask;
  tp.desc = p.tdesc_row;
  tp.grp_ptr = p.trow_ptr;
  tp.n_grp = p.n_trows;
  tp.N = p.N;
  tp.H = H;
  tp.qmul = f.qmul;
  tp.lse = lse;
  tp.err = p.err;
  return launch_tile_fwd(tp, D, p.num_sms, st);
}

static gattn_status bwd_common(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                               const void* Q, const void* K, const void* V,
                               const gattn_score* score, const void* dout, const float* lse,
                               void* workspace, size_t workspace_bytes, BwdParams* b, int* rb,
                               Workspace* w) {
  GATTN_REQUIRE(plan, GATTN_ERR_INVALID_ARG, "plan is NULL");
  gattn_status s = check_shape(H, D, dtype, rb);
  if (s != GATTN_OK) return s;
  if ((s = check_score(score, D, &b->qmul, &b->scale, &b->slope)) != GATTN_OK) return s;
  if (plan->p.N == 0) return GATTN_OK;
  if ((s = check_tensor(Q, "Q")) || (s = check_tensor(K, "K")) || (s = check_tensor(V, "V")) ||
      (s = check_tensor(dout, "dout")))
    return s;
  GATTN_REQUIRE(lse && aligned(lse, 4), GATTN_ERR_INVALID_ARG, "lse must be a device pointer");
  *w = ws_layout(plan->p, H, D);
  GATTN_REQUIRE(workspace && aligned(workspace, 16) && workspace_bytes >= w->total,
                GATTN_ERR_INVALID_ARG, "workspace needs %zu bytes (16-byte aligned), got %zu",
                w->total, workspace_bytes);
  char* ws = static_cast<char*>(workspace);
  b->Q = Q;
  b->K = K;
  b->V = V;
  b->dO = dout;
  b->lse = lse;
  b->delta = reinterpret_cast<float*>(ws + w->delta);
  b->a = score->a;
  b->H = H;
  b->D = D;
  b->rows16 = (H % 4 == 0) && aligned(lse, 16);
  b->da_part = reinterpret_cast<float*>(ws + w->da_part);
  b->da_cnt = plan->p.cnt_da;
  b->err = plan->p.err;
  b->fail_first_wait = plan->p.fail_first_wait;
  return GATTN_OK;
}

gattn_status gattn_bwd_dq(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                          const void* Q, const void* K, const void* V, const gattn_score* score,
                          const void* out, const void* dout, const float* lse, void* dQ,
                          float* da, void* workspace, size_t workspace_bytes,
                          gattn_stream_t stream) {
  BwdParams b{};
  int rb = 0;
  Workspace w{};
  gattn_status s = bwd_common(plan, H, D, dtype, Q, K, V, score, dout, lse, workspace,
                              workspace_bytes, &b, &rb, &w);
  if (s != GATTN_OK) return s;
  const Plan& p = plan->p;
  const bool gat = score->kind == GATTN_SCORE_GATV2;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (p.N == 0) {
    if (gat && da) {
      const cudaError_t e = cudaMemsetAsync(da, 0, size_t(H) * D * sizeof(float), st);
      GATTN_REQUIRE(e == cudaSuccess, GATTN_ERR_CUDA, "cudaMemsetAsync failed");
    }
    return GATTN_OK;
  }
  if ((s = check_tensor(out, "out")) || (s = check_tensor(dQ, "dQ"))) return s;
  GATTN_REQUIRE(!gat || !da || aligned(da, 4), GATTN_ERR_INVALID_ARG, "da misaligned");
  // dense tiles on the tensor cores: the CSR pass covers the residual edges
  // (and writes Delta for every node), the tile pass adds the tiles' dQ
  const bool tiles = tile_path(p, dtype, score->kind, D);
  b.O = out;
  b.items = tiles ? p.items_r : p.items;
  b.sorted = tiles ? p.sorted_r : p.sorted;
  b.n_items = tiles ? p.n_chunks_r + p.n_light_r : p.n_chunks + p.n_light;
  b.n_chunks = tiles ? p.n_chunks_r : p.n_chunks;
  b.N = p.N;
  {
    const int es = (int)dtype_size(dtype);
    const bool bf = dtype == GATTN_BF16;
    const int64_t HD = int64_t(H) * D;
    if (!encode_rows_map(&b.mi0, Q, es, bf, p.N, HD) ||
        !encode_rows_map(&b.mi1, dout, es, bf, p.N, HD) ||
        !encode_rows_map(&b.mi2, out, es, bf, p.N, HD) ||
        !encode_rows_map(&b.me0, K, es, bf, p.N, HD) || !encode_rows_map(&b.me1, V, es, bf, p.N, HD) ||
        (b.rows16 && !encode_rows_map(&b.ms0, lse, 4, false, p.N, H)))
      return GATTN_ERR_CUDA;
  }
  b.idx = tiles ? p.indices_r : p.indices;
  b.G1 = dQ;
  b.G2 = nullptr;
  b.da = gat ? da : nullptr;
  b.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.dq_part);
  b.tree = tiles ? Tree{p.parent_r, p.kids_r, p.n_chunks_r, p.cnt_dq_r}
                 : Tree{p.parent, p.kids, p.n_chunks, p.cnt_dq};
  if ((s = launch_bwd_csr(dtype, rb, D * (int)dtype_size(dtype), score->kind,
                          stage_bytes(tiles ? p.M_res : p.M, b.n_items), b, p.num_sms, st,
                          nullptr)) != GATTN_OK)
    return s;
  if ((s = launched("backward (CSR pass)")) != GATTN_OK || !tiles) return s;
  TileBwdParams tp{};
  const int64_t HD = int64_t(H) * D;
  if (!encode_tile_map(&tp.ma0, Q, p.N, HD) || !encode_tile_map(&tp.ma1, dout, p.N, HD) ||
      !encode_tile_map(&tp.mb0, K, p.N, HD) || !encode_tile_map(&tp.mb1, V, p.N, HD) ||
      !encode_tile_map(&tp.mg1, dQ, p.N, HD))
    return GATTN_ERR_CUDA;
  tp.mask = p.tile_mask;
  tp.desc = p.tdesc_row;
  tp.grp_ptr = p.trow_ptr;
  tp.n_grp = p.n_trows;
  tp.N = p.N;
  tp.H = H;
  tp.qmul = b.qmul;
  tp.scale = b.scale;
  tp.lse = lse;
  tp.delta = b.delta;
  tp.g1 = dQ;
  tp.g2 = nullptr;
  tp.err = p.err;
  return launch_tile_bwd(tp, D, false, p.num_sms, st);
}

gattn_status gattn_bwd_dkdv(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                            const void* Q, const void* K, const void* V,
                            const gattn_score* score, const void* dout, const float* lse,
                            void* dK, void* dV, void* workspace, size_t workspace_bytes,
                            gattn_stream_t stream) {
  BwdParams b{};
  int rb = 0;
  Workspace w{};
  gattn_status s = bwd_common(plan, H, D, dtype, Q, K, V, score, dout, lse, workspace,
                              workspace_bytes, &b, &rb, &w);
  if (s != GATTN_OK) return s;
  const Plan& p = plan->p;
  if (p.N == 0) return GATTN_OK;
  if ((s = check_tensor(dK, "dK")) || (s = check_tensor(dV, "dV"))) return s;
  // dense tiles: the CSC pass covers the residual edges, the tile pass adds
  const bool tiles = tile_path(p, dtype, score->kind, D);
  b.items = tiles ? p.items_src_r : p.items_src;
  b.sorted = tiles ? p.sorted_src_r : p.sorted_src;
  b.n_items = tiles ? p.n_chunks_src_r + p.n_light_src_r : p.n_src_chunks + p.n_light_src;
  b.n_chunks = tiles ? p.n_chunks_src_r : p.n_src_chunks;
  b.N = p.N;
  {
    const int es = (int)dtype_size(dtype);
    const bool bf = dtype == GATTN_BF16;
    const int64_t HD = int64_t(H) * D;
    if (!encode_rows_map(&b.mi0, K, es, bf, p.N, HD) || !encode_rows_map(&b.mi1, V, es, bf, p.N, HD) ||
        !encode_rows_map(&b.me0, Q, es, bf, p.N, HD) ||
        !encode_rows_map(&b.me1, dout, es, bf, p.N, HD))
      return GATTN_ERR_CUDA;
  }
  b.idx = tiles ? p.csc_dst_r : p.csc_dst;
  b.G1 = dK;
  b.G2 = dV;
  b.da = nullptr;
  b.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.dkv_part);
  b.tree = tiles ? Tree{p.parent_src_r, p.kids_src_r, p.n_chunks_src_r, p.cnt_dkv_r}
                 : Tree{p.parent_src, p.kids_src, p.n_src_chunks, p.cnt_dkv};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = launch_bwd_csc(dtype, rb, D * (int)dtype_size(dtype), score->kind,
                          stage_bytes(tiles ? p.M_res : p.M, b.n_items), b, p.num_sms, st,
                          nullptr)) != GATTN_OK)
    return s;
  if ((s = launched("backward (CSC pass)")) != GATTN_OK || !tiles) return s;
  TileBwdParams tp{};
  const int64_t HD = int64_t(H) * D;
  if (!encode_tile_map(&tp.ma0, K, p.N, HD) || !encode_tile_map(&tp.ma1, V, p.N, HD) ||
      !encode_tile_map(&tp.mb0, Q, p.N, HD) || !encode_tile_map(&tp.mb1, dout, p.N, HD) ||
      !encode_tile_map(&tp.mg1, dK, p.N, HD) || !encode_tile_map(&tp.mg2, dV, p.N, HD))
    return GATTN_ERR_CUDA;
  tp.mask = p.tile_mask_t;
  tp.desc = p.tdesc_col;
  tp.grp_ptr = p.tcol_ptr;
  tp.n_grp = p.n_tcols;
  tp.N = p.N;
  tp.H = H;
  tp.qmul = b.qmul;
  tp.scale = b.scale;
  tp.lse = lse;
  tp.delta = b.delta;
  tp.g1 = dK;
  tp.g2 = dV;
  tp.err = p.err;
  return launch_tile_bwd(tp, D, true, p.num_sms, st);
}

gattn_status gattn_bwd(const gattn_plan* plan, int32_t H, int32_t D, gattn_dtype dtype,
                       const void* Q, const void* K, const void* V, const gattn_score* score,
                       const void* out, const void* dout, const float* lse, void* dQ, void* dK,
                       void* dV, float* da, void* workspace, size_t workspace_bytes,
                       gattn_stream_t stream) {
  gattn_status s = gattn_bwd_dq(plan, H, D, dtype, Q, K, V, score, out, dout, lse, dQ, da,
                                workspace, workspace_bytes, stream);
  if (s != GATTN_OK) return s;
  return gattn_bwd_dkdv(plan, H, D, dtype, Q, K, V, score, dout, lse, dK, dV, workspace,
                        workspace_bytes, stream);
}

}  // extern "C"
