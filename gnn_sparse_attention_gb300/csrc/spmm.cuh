// spmm.cuh -- weighted sparse-dense products of the adjacency (GCN-style
// aggregation).
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", SpMM-based convolutions (GCN,
// GraphConv: H' = A H W): graph metadata is built once and cached, the
// transposed adjacency is precomputed for the backward, and a weighted
// block-sparse (WSB) form of locally dense neighbourhoods runs on the tensor
// cores.
//
// spmm_kernel: y[i] = sum over the edges e of item i of w[e] x[src(e)], on
// the plan's work items -- the CSR items for y = A x, the cached CSC items
// for y = A^T x (the backward dX = A^T dY).  The x rows come through the
// attention kernels' gather pipeline (attn_pipe.cuh); each group keeps fp32
// sums in registers; heavy chunks add their partial rows up the node's merge
// tree in chunk order (deterministic).  The tile part of the WSB path lives
// in spmm_tile.cu.
#pragma once

#include "attn_pipe.cuh"

namespace gattn {

struct SpmmParams {
  CUtensorMap mx;        // row-gather map of x
  const int4* sorted;    // items by decreasing length
  int64_t n_items;
  int64_t n_chunks;      // items [0, n_chunks) are heavy chunks
  int N, F;
  const int32_t* idx;    // sources per edge position (CSR indices or CSC destinations)
  const float* w;        // weight per edge position, same order as idx
  void* y;               // [N, F] in the I/O dtype
  float* part;           // [slots][F] partial rows of heavy nodes
  Tree tree;
  int32_t* err;
};

template <typename T, int RB, int SB>
struct SpmmShape {
  using L = Lay<T, RB, SB>;
  static constexpr int STAGE = L::B * RB;
  static constexpr int WARP_BYTES = align128(kStages * STAGE + L::META);
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

template <typename T, int RB, int SB>
__global__ void __launch_bounds__(SpmmShape<T, RB, SB>::THREADS) spmm_kernel(const __grid_constant__ SpmmParams p) {
  using L = Lay<T, RB, SB>;
  using Sh = SpmmShape<T, RB, SB>;
  using PR = Pairs<T>;
  constexpr int NC = L::NC, TPR = L::TPR, G = L::G, SE = L::SE, B = L::B, S = kStages;
  constexpr int PP = PR::P;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int g = lane / TPR, t = lane % TPR;
  Ring<L, Sh::STAGE> ring;
  ring.init(smem + (threadIdx.x >> 5) * Sh::WARP_BYTES, lane);
  int elem[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) elem[c] = (t * NC + c) * (16 / (int)sizeof(T));

  const int64_t warp = (int64_t(blockIdx.x) * Sh::THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * Sh::THREADS) >> 5;
  BundleCursor<G, SE> cur;
  cur.start(p.sorted, p.n_items, p.idx, p.N, warp, nwarps, ring.items, lane);

  auto issue = [&](int s) {
    if (lane == 0) {
      const int4* dsc = ring.desc_at(s);
      if (dsc[0].x != -3) {
        uint8_t* st = ring.stage_at(s);
        uint64_t* bar = ring.bar_at(s);
        fence_proxy_async();
        mbar_expect_tx(bar, (B / 4) * L::SET_BYTES);
#pragma unroll
        for (int b4 = 0; b4 < B / 4; ++b4) {
          const int4 r = ring.eset(s, b4);
          L::gather(st, 4 * b4, &p.mx, r.x, r.y, r.z, r.w, bar);
        }
      }
    }
    __syncwarp();
    cp_async_commit();
  };

  for (int s = 0; s < S; ++s) ring.generate(cur, s, lane);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int s = 0; s < S - 1; ++s) {
    ring.generate(cur, S + s, lane);
    issue(s);
  }

  float2 acc[NC][PP];
  for (int i = 0;; ++i) {
    ring.generate(cur, i + 2 * S - 1, lane);
    __syncwarp();
    issue(i + S - 1);
    cp_async_wait<S - 1>();
    __syncwarp();
    const int4* dsc = ring.desc_at(i);
    if (dsc[0].x == -3) break;
    if (!__all_sync(FULL, ring.wait_rows(i, p.err, lane))) break;
    const int4 d = dsc[g];
    const bool act = d.x >= 0;
    const int cnt = act ? (d.z & kCntMask) : 0;
    const uint8_t* st = ring.stage_at(i);
    if (act && (d.z & kFirst)) {
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int v = 0; v < PP; ++v) acc[c][v] = f2s(0.f);
    }
    for (int k = 0; k < cnt; ++k) {
      const float we = __ldg(p.w + d.w + k);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float2 xf[PP];
        PR::load(lds16(st + L::off(g * SE + k, (t * NC + c) * 16)), xf);
#pragma unroll
        for (int v = 0; v < PP; ++v) acc[c][v] = f2fma(f2s(we), xf[v], acc[c][v]);
      }
    }

    const bool fin = act && (d.z & kLast);
    const bool heavy = fin && d.y < p.n_chunks;
    bool write = fin && !heavy;
    if (heavy) {
      auto store = [&](int slot) {
        float* pb = p.part + int64_t(slot) * p.F;
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; v += 2)
            *reinterpret_cast<float4*>(pb + elem[c] + 2 * v) =
                make_float4(acc[c][v].x, acc[c][v].y, acc[c][v + 1].x, acc[c][v + 1].y);
      };
      auto merge = [&](int c0, int cn) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; ++v) acc[c][v] = f2s(0.f);
        for (int kk = 0; kk < cn; ++kk) {
          const float* pc = p.part + int64_t(c0 + kk) * p.F;
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int v = 0; v < PP / 2; ++v) {
              const float4 f = __ldcg(reinterpret_cast<const float4*>(pc + elem[c] + 4 * v));
              acc[c][2 * v].x += f.x;
              acc[c][2 * v].y += f.y;
              acc[c][2 * v + 1].x += f.z;
              acc[c][2 * v + 1].y += f.w;
            }
        }
      };
      write = climb(p.tree, d.y, group_mask<TPR>(g), g * TPR, t == 0, merge, store);
    }
    if (write) {
      char* yb = static_cast<char*>(p.y) + int64_t(d.x) * RB;
#pragma unroll
      for (int c = 0; c < NC; ++c) *reinterpret_cast<uint4*>(yb + (t * NC + c) * 16) = PR::store(acc[c]);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  ring.release(lane);
}

// Launch for one (dtype, row bytes) with run-time stage bytes.
template <typename T, int RB>
gattn_status spmm_dispatch(int sb, const SpmmParams& p, int num_sms, cudaStream_t st) {
  auto go = [&](auto kern, int threads, int warps, int smem, int* cache) -> gattn_status {
    int bps = *cache;
    if (bps == 0) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, threads, smem) != cudaSuccess ||
          bps < 1)
        bps = 1;
      if (bps > kMaxBlocksPerSm) bps = kMaxBlocksPerSm;
      *cache = bps;
    }
    const int64_t need = ((p.n_items + kUnit - 1) / kUnit + warps - 1) / warps;
    int64_t grid = int64_t(num_sms) * bps;
    if (grid > need) grid = need;
    kern<<<int(grid < 1 ? 1 : grid), threads, smem, st>>>(p);
    return GATTN_OK;
  };
  static int cache[2] = {0, 0};
  if (sb == 4096) {
    using Sh = SpmmShape<T, RB, 4096>;
    return go(spmm_kernel<T, RB, 4096>, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[0]);
  }
  using Sh = SpmmShape<T, RB, 8192>;
  return go(spmm_kernel<T, RB, 8192>, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[1]);
}

#define GATTN_DECLARE_SPMM(TNAME, RB_) \
  gattn_status launch_spmm_##TNAME##_##RB_(int sb, const SpmmParams& p, int num_sms, cudaStream_t st);
#define GATTN_FOR_SPMM_ROWS(X, TNAME) \
  X(TNAME, 32) X(TNAME, 64) X(TNAME, 128) X(TNAME, 256) X(TNAME, 512) X(TNAME, 1024) X(TNAME, 2048)
GATTN_FOR_SPMM_ROWS(GATTN_DECLARE_SPMM, f32)
GATTN_FOR_SPMM_ROWS(GATTN_DECLARE_SPMM, bf16)

// WSB tile part: y[rows of each row block with tiles] += sum over its tiles
// W_t x[cols]; W_t are bf16 [128 x 128] weight tiles.  F a multiple of 64,
// at most 512.  Runs after spmm_kernel wrote the residual part of y.
struct WsbParams {
  CUtensorMap mw;              // weight tiles as [n_tiles * 128, 128] bf16, 64 x 128 boxes
  CUtensorMap mx;              // x as [N, F] bf16, 64 x 128 boxes
  CUtensorMap my;              // y the same way (residual result in, sum out)
  const int32_t* tile_cb;
  const int32_t* trow_rb;
  const int32_t* trow_ptr;
  int64_t n_trows;
  int N, F;
  void* y;                     // bf16 [N, F]
  int32_t* err;
};
gattn_status launch_wsb_tiles(const WsbParams& p, cudaStream_t st);

}  // namespace gattn
