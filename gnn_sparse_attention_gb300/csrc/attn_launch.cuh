// attn_launch.cuh -- template instantiation and launch of the attention
// kernels for one I/O dtype.  Each including .cu file defines GATTN_T (the
// element type) and GATTN_SUFFIX and gets the three launchers for every
// supported row size (32 .. 2048 bytes) and both score kinds.
#pragma once

#include "attn_bwd.cuh"
#include "attn_fwd.cuh"

namespace gattn {

// Grid of a persistent kernel: every SM gets as many 256-thread blocks as fit
// (capped at kMaxBlocksPerSm), but never more blocks than work items need.
template <typename Kern>
int persistent_grid(Kern kernel, int num_sms, int64_t n_items) {
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, kThreads, 0) != cudaSuccess ||
      bps < 1)
    bps = 1;
  if (bps > kMaxBlocksPerSm) bps = kMaxBlocksPerSm;
  const int64_t need = (n_items + kWarpsPerBlock - 1) / kWarpsPerBlock;
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
    auto k = kind == GATTN_SCORE_DOT ? fwd_kernel<T, RB_, GATTN_SCORE_DOT>         \
                                     : fwd_kernel<T, RB_, GATTN_SCORE_GATV2>;      \
    const int g = persistent_grid(k, num_sms, p.n_items);                          \
    if (grid_out) *grid_out = g;                                                   \
    k<<<g, kThreads, 0, st>>>(p);                                                  \
    return GATTN_OK;                                                               \
  }
    switch (rb) { GATTN_RB_CASES(GATTN_FWD_CASE) default: return GATTN_ERR_UNSUPPORTED; }
#undef GATTN_FWD_CASE
  }
  static gattn_status bwd_csr(int rb, int kind, const BwdParams& p, int num_sms, cudaStream_t st,
                              int* grid_out) {
#define GATTN_CSR_CASE(RB_)                                                         \
  case RB_: {                                                                       \
    auto k = kind == GATTN_SCORE_DOT ? bwd_csr_kernel<T, RB_, GATTN_SCORE_DOT>      \
                                     : bwd_csr_kernel<T, RB_, GATTN_SCORE_GATV2>;   \
    const int g = persistent_grid(k, num_sms, p.n_items);                           \
    if (grid_out) *grid_out = g;                                                    \
    k<<<g, kThreads, 0, st>>>(p);                                                   \
    return GATTN_OK;                                                                \
  }
    switch (rb) { GATTN_RB_CASES(GATTN_CSR_CASE) default: return GATTN_ERR_UNSUPPORTED; }
#undef GATTN_CSR_CASE
  }
  static gattn_status bwd_csc(int rb, int kind, const BwdParams& p, int num_sms, cudaStream_t st,
                              int* grid_out) {
#define GATTN_CSC_CASE(RB_)                                                         \
  case RB_: {                                                                       \
    auto k = kind == GATTN_SCORE_DOT ? bwd_csc_kernel<T, RB_, GATTN_SCORE_DOT>      \
                                     : bwd_csc_kernel<T, RB_, GATTN_SCORE_GATV2>;   \
    const int g = persistent_grid(k, num_sms, p.n_items);                           \
    if (grid_out) *grid_out = g;                                                    \
    k<<<g, kThreads, 0, st>>>(p);                                                   \
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
