// attn_launch.cuh -- template instantiation and launch of the attention
// kernels for one I/O dtype.  Each including .cu file defines GATTN_T (the
// element type) and GATTN_SUFFIX and gets the three launchers for every
// supported row size (32 .. 2048 bytes) and both score kinds.
#pragma once

#include "attn_bwd.cuh"
#include "attn_fwd.cuh"

namespace gattn {

// Blocks per SM of a persistent kernel with `smem` bytes of dynamic shared
// memory (the attribute that allows more than 48 KB is set on first use).
// Cached per kernel: the first call of each instantiation does the queries.
template <typename Kern>
int blocks_per_sm(Kern kernel, int threads, int smem, int* cache) {
  if (*cache > 0) return *cache;
  int bps = 0;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, threads, smem) != cudaSuccess ||
      bps < 1)
    bps = 1;
  if (bps > kMaxBlocksPerSm) bps = kMaxBlocksPerSm;
  *cache = bps;
  return bps;
}

// Grid of a persistent kernel: every SM gets as many blocks as fit, but
// never more blocks than there are work items for their warps.
inline int persistent_grid(int bps, int warps_per_block, int num_sms, int64_t n_items) {
  const int64_t need = (n_items + warps_per_block - 1) / warps_per_block;
  int64_t g = int64_t(num_sms) * bps;
  if (g > need) g = need;
  return (int)(g < 1 ? 1 : g);
}

#define GATTN_RB_CASES(X) X(32) X(64) X(128) X(256) X(512) X(1024) X(2048)

template <typename T>
struct Launch {
  static gattn_status fwd(int rb, int kind, const FwdParams& p, int num_sms, cudaStream_t st,
                          int* grid_out) {
#define GATTN_FWD_CASE(RB_)                                                        \
  case RB_: {                                                                      \
    using Sh = FwdShape<T, RB_>;                                                          \
    static int cache[2] = {0, 0};                                                    \
    auto k = kind == GATTN_SCORE_DOT ? fwd_kernel<T, RB_, GATTN_SCORE_DOT>                    \
                                     : fwd_kernel<T, RB_, GATTN_SCORE_GATV2>;                 \
    const int bps = blocks_per_sm(k, Sh::THREADS, Sh::SMEM, &cache[kind != 0]);       \
    const int g = persistent_grid(bps, Sh::WARPS, num_sms, (p.n_items + kUnit - 1) / kUnit);               \
    if (grid_out) *grid_out = g;                                                     \
    k<<<g, Sh::THREADS, Sh::SMEM, st>>>(p);                                          \
    return GATTN_OK;                                                               \
  }
    switch (rb) { GATTN_RB_CASES(GATTN_FWD_CASE) default: return GATTN_ERR_UNSUPPORTED; }
#undef GATTN_FWD_CASE
  }
  static gattn_status bwd_csr(int rb, int kind, const BwdParams& p, int num_sms, cudaStream_t st,
                              int* grid_out) {
#define GATTN_CSR_CASE(RB_)                                                         \
  case RB_: {                                                                       \
    using Sh = CsrShape<T, RB_>;                                                          \
    static int cache[2] = {0, 0};                                                    \
    auto k = kind == GATTN_SCORE_DOT ? bwd_csr_kernel<T, RB_, GATTN_SCORE_DOT>                    \
                                     : bwd_csr_kernel<T, RB_, GATTN_SCORE_GATV2>;                 \
    const int bps = blocks_per_sm(k, Sh::THREADS, Sh::SMEM, &cache[kind != 0]);       \
    const int g = persistent_grid(bps, Sh::WARPS, num_sms, (p.n_items + kUnit - 1) / kUnit);               \
    if (grid_out) *grid_out = g;                                                     \
    k<<<g, Sh::THREADS, Sh::SMEM, st>>>(p);                                          \
    return GATTN_OK;                                                                \
  }
    switch (rb) { GATTN_RB_CASES(GATTN_CSR_CASE) default: return GATTN_ERR_UNSUPPORTED; }
#undef GATTN_CSR_CASE
  }
  static gattn_status bwd_csc(int rb, int kind, const BwdParams& p, int num_sms, cudaStream_t st,
                              int* grid_out) {
#define GATTN_CSC_CASE(RB_)                                                         \
  case RB_: {                                                                       \
    using Sh = CscShape<T, RB_>;                                                          \
    static int cache[2] = {0, 0};                                                    \
    auto k = kind == GATTN_SCORE_DOT ? bwd_csc_kernel<T, RB_, GATTN_SCORE_DOT>                    \
                                     : bwd_csc_kernel<T, RB_, GATTN_SCORE_GATV2>;                 \
    const int bps = blocks_per_sm(k, Sh::THREADS, Sh::SMEM, &cache[kind != 0]);       \
    const int g = persistent_grid(bps, Sh::WARPS, num_sms, (p.n_items + kUnit - 1) / kUnit);               \
    if (grid_out) *grid_out = g;                                                     \
    k<<<g, Sh::THREADS, Sh::SMEM, st>>>(p);                                          \
    return GATTN_OK;                                                                \
  }
    switch (rb) { GATTN_RB_CASES(GATTN_CSC_CASE) default: return GATTN_ERR_UNSUPPORTED; }
#undef GATTN_CSC_CASE
  }
};

// Entry points implemented by attn_f32.cu / attn_bf16.cu.
gattn_status launch_fwd(gattn_dtype dt, int rb, int kind, const FwdParams& p, int num_sms,
                        cudaStream_t st, int* grid_out);
gattn_status launch_bwd_csr(gattn_dtype dt, int rb, int kind, const BwdParams& p, int num_sms,
                            cudaStream_t st, int* grid_out);
gattn_status launch_bwd_csc(gattn_dtype dt, int rb, int kind, const BwdParams& p, int num_sms,
                            cudaStream_t st, int* grid_out);

}  // namespace gattn
