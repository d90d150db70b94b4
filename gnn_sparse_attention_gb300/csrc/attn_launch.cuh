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

// One (row bytes, head bytes, stage bytes) instantiation of a kernel; head
// bytes DB = D * sizeof(T) in {16, ..., 512} and never above the row.
template <typename T, int RB, int DB, int SB>
struct Case {
  static constexpr bool ok = DB <= RB;

  static gattn_status fwd(int kind, const FwdParams& p, int num_sms, cudaStream_t st, int* g) {
    if constexpr (!ok) {
      return GATTN_ERR_UNSUPPORTED;
    } else {
      using Sh = FwdShape<T, RB, SB>;
      static int cache[2] = {0, 0};
      auto k = kind == GATTN_SCORE_DOT ? fwd_kernel<T, RB, DB, GATTN_SCORE_DOT, SB>
                                       : fwd_kernel<T, RB, DB, GATTN_SCORE_GATV2, SB>;
      return go(k, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[kind != 0], p, num_sms, st, g);
    }
  }
  static gattn_status csr(int kind, const BwdParams& p, int num_sms, cudaStream_t st, int* g) {
    if constexpr (!ok) {
      return GATTN_ERR_UNSUPPORTED;
    } else {
      using Sh = CsrShape<T, RB, SB>;
      static int cache[2] = {0, 0};
      auto k = kind == GATTN_SCORE_DOT ? bwd_csr_kernel<T, RB, DB, GATTN_SCORE_DOT, SB>
                                       : bwd_csr_kernel<T, RB, DB, GATTN_SCORE_GATV2, SB>;
      return go(k, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[kind != 0], p, num_sms, st, g);
    }
  }
  static gattn_status csc(int kind, const BwdParams& p, int num_sms, cudaStream_t st, int* g) {
    if constexpr (!ok) {
      return GATTN_ERR_UNSUPPORTED;
    } else {
      using Sh = CscShape<T, RB, SB, DB>;
      static int cache[2] = {0, 0};
      auto k = kind == GATTN_SCORE_DOT ? bwd_csc_kernel<T, RB, DB, GATTN_SCORE_DOT, SB>
                                       : bwd_csc_kernel<T, RB, DB, GATTN_SCORE_GATV2, SB>;
      return go(k, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[kind != 0], p, num_sms, st, g);
    }
  }

  template <typename Kern, typename P>
  static gattn_status go(Kern k, int threads, int warps, int smem, int* cache, const P& p,
                         int num_sms, cudaStream_t st, int* g) {
    const int bps = blocks_per_sm(k, threads, smem, cache);
    const int grid = persistent_grid(bps, warps, num_sms, (p.n_items + kUnit - 1) / kUnit);
    if (g) *g = grid;
    k<<<grid, threads, smem, st>>>(p);
    return GATTN_OK;
  }
};

// Runtime dispatch over the head bytes for one row size and stage size.
template <typename T, int RB, int SB, int PASS, typename P>
gattn_status dispatch_db(int db, int kind, const P& p, int num_sms, cudaStream_t st, int* g) {
#define GATTN_DB_CASE(DB_)                                                     \
  case DB_:                                                                    \
    if constexpr (PASS == 0) return Case<T, RB, DB_, SB>::fwd(kind, p, num_sms, st, g); \
    else if constexpr (PASS == 1) return Case<T, RB, DB_, SB>::csr(kind, p, num_sms, st, g); \
    else return Case<T, RB, DB_, SB>::csc(kind, p, num_sms, st, g);
  switch (db) {
    GATTN_DB_CASE(16)
    GATTN_DB_CASE(32)
    GATTN_DB_CASE(64)
    GATTN_DB_CASE(128)
    GATTN_DB_CASE(256)
    GATTN_DB_CASE(512)
    default:
      return GATTN_ERR_UNSUPPORTED;
  }
#undef GATTN_DB_CASE
}

// Stage bytes of the gather pipeline: short work items (mean edge count at
// most kShortItem) waste fewer edge slots in small stages; long ones pay
// the per-stage overhead less often in large stages.
constexpr int kStageSmall = 4096;
constexpr int kStageLarge = 8192;
constexpr double kShortItem = 16.0;
inline int stage_bytes(int64_t edges, int64_t items) {
  return items > 0 && double(edges) / double(items) <= kShortItem ? kStageSmall : kStageLarge;
}

// Launchers for one (pass, dtype, row size, stage size); each lives in its
// own translation unit (k_<pass>_<dtype>_<row bytes>_<stage bytes>.cu) so the
// library builds in parallel.  PASS: 0 forward, 1 backward CSR pass, 2
// backward CSC pass.
#define GATTN_DECLARE_LAUNCHER(PASS_NAME, PT, TNAME, RB_, SB_)                           \
  gattn_status launch_##PASS_NAME##_##TNAME##_##RB_##_##SB_(int db, int kind, const PT& p, \
                                                            int num_sms, cudaStream_t st, int* g);
#define GATTN_FOR_ROWS_SB(X, PASS_NAME, PT, TNAME, SB_)                                   \
  X(PASS_NAME, PT, TNAME, 32, SB_) X(PASS_NAME, PT, TNAME, 64, SB_)                       \
  X(PASS_NAME, PT, TNAME, 128, SB_) X(PASS_NAME, PT, TNAME, 256, SB_)                     \
  X(PASS_NAME, PT, TNAME, 512, SB_) X(PASS_NAME, PT, TNAME, 1024, SB_)                    \
  X(PASS_NAME, PT, TNAME, 2048, SB_)
#define GATTN_FOR_ROWS(X, PASS_NAME, PT, TNAME)     \
  GATTN_FOR_ROWS_SB(X, PASS_NAME, PT, TNAME, 4096) \
  GATTN_FOR_ROWS_SB(X, PASS_NAME, PT, TNAME, 8192)
GATTN_FOR_ROWS(GATTN_DECLARE_LAUNCHER, fwd, FwdParams, f32)
GATTN_FOR_ROWS(GATTN_DECLARE_LAUNCHER, fwd, FwdParams, bf16)
GATTN_FOR_ROWS(GATTN_DECLARE_LAUNCHER, csr, BwdParams, f32)
GATTN_FOR_ROWS(GATTN_DECLARE_LAUNCHER, csr, BwdParams, bf16)
GATTN_FOR_ROWS(GATTN_DECLARE_LAUNCHER, csc, BwdParams, f32)
GATTN_FOR_ROWS(GATTN_DECLARE_LAUNCHER, csc, BwdParams, bf16)

// sb: stage bytes (kStageSmall or kStageLarge, see stage_bytes)
gattn_status launch_fwd(gattn_dtype dt, int rb, int db, int kind, int sb, const FwdParams& p,
                        int num_sms, cudaStream_t st, int* grid_out);
gattn_status launch_bwd_csr(gattn_dtype dt, int rb, int db, int kind, int sb, const BwdParams& p,
                            int num_sms, cudaStream_t st, int* grid_out);
gattn_status launch_bwd_csc(gattn_dtype dt, int rb, int db, int kind, int sb, const BwdParams& p,
                            int num_sms, cudaStream_t st, int* grid_out);

}  // namespace gattn
