// pool.cuh -- degree-aware max / min pooling over the in-neighbours.
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", reduction-based layers: a per-edge
// message followed by a neighbourhood reduction (min / max pooling), which
// is sensitive to the degree distribution; nodes are split by a degree
// threshold into light nodes (one feature-parallel pass each) and heavy
// nodes tiled over edge chunks reduced in parallel, the chunk results merged
// with atomic operations on packed (value, index) pairs so that heavy-tailed
// degrees need no extra memory.
//
// Here the message of edge j -> i is the source row x[j]; the result is
// out[i][f] = max_j x[j][f] (min for GATTN_POOL_MIN) and arg[i][f] = the
// smallest source id attaining it (a node without in-edges: out 0, arg -1).
//
// Forward: the attention kernels' gather pipeline (attn_pipe.cuh) streams
// the x rows of every work item of the plan; each lane keeps the running
// best value and source of its elements in registers.  A light item writes
// its row; a heavy chunk folds its row into the node's packed 64-bit
// (order-preserving value key, complemented source id) words with
// atomicMax -- largest value, then smallest id, whatever the arrival order
// -- and the chunk that arrives last (an arrival counter per heavy node)
// takes the words back (atomicExch to zero, ready for the next call) and
// writes the node's row.
//
// Backward: dx[j][f] = sum of dout[i][f] over the nodes i with arg[i][f] ==
// j -- an O(N * F) scatter (fp32 atomics into a workspace accumulator, then
// one pass that rounds to the I/O dtype), independent of M.
#pragma once

#include "attn_pipe.cuh"

namespace gattn {

struct PoolParams {
  CUtensorMap mx;               // row-gather map of x
  const int4* sorted;           // items by decreasing length
  const int4* items;            // plan items (w = heavy id of a chunk)
  const int32_t* hfirst;        // [n_heavy + 1] first chunk of each heavy node
  int64_t n_items;
  int64_t n_chunks;             // items [0, n_chunks) are heavy chunks
  int N, F;
  const int32_t* idx;           // CSR sources
  void* out;                    // [N, F] in the I/O dtype
  int32_t* arg;                 // [N, F]
  unsigned long long* packed;   // [n_heavy, F] zero before the call
  int32_t* cnt;                 // [n_heavy] zero before the call
  int32_t* err;
};

template <typename T, int RB, int SB>
struct PoolShape {
  using L = Lay<T, RB, SB>;
  static constexpr int STAGE = L::B * RB;  // the stage's source rows
  static constexpr int WARP_BYTES = align128(kStages * STAGE + L::META);
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

// Order-preserving 32-bit key of a float (-0 and +0 share a key) and back.
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <typename T, int RB, int SB, int OP>
__global__ void __launch_bounds__(PoolShape<T, RB, SB>::THREADS) pool_fwd_kernel(const __grid_constant__ PoolParams p) {
  using L = Lay<T, RB, SB>;
  using Sh = PoolShape<T, RB, SB>;
  constexpr int NC = L::NC, TPR = L::TPR, G = L::G, SE = L::SE, B = L::B, S = kStages;
  constexpr int VEC = L::VEC;  // elements per 16-byte chunk
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int NONE = 0x7fffffff;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int g = lane / TPR, t = lane % TPR;
  Ring<L, Sh::STAGE> ring;
  ring.init(smem + (threadIdx.x >> 5) * Sh::WARP_BYTES, lane);

  const int64_t warp = (int64_t(blockIdx.x) * Sh::THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * Sh::THREADS) >> 5;
  BundleCursor<G, SE> cur;
  cur.start(p.sorted, p.n_items, p.idx, p.N, warp, nwarps, ring.items, lane);

  // the stage's source rows by TMA gathers from lane 0 (pad row N in unused slots)
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

  float best[NC][VEC];
  int who[NC][VEC];
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
    const int* ix = ring.ix_at(i);
    if (act && (d.z & kFirst)) {
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          best[c][e] = OP == 0 ? neg_inf() : -neg_inf();
          who[c][e] = NONE;
        }
    }
    for (int k = 0; k < cnt; ++k) {
      const int j = ix[g * SE + k];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 u = lds16(st + L::off(g * SE + k, (t * NC + c) * 16));
        float v[VEC];
        if constexpr (sizeof(T) == 2) {
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(w[q] << 16);
            v[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
          }
        } else {
          v[0] = __uint_as_float(u.x);
          v[1] = __uint_as_float(u.y);
          v[2] = __uint_as_float(u.z);
          v[3] = __uint_as_float(u.w);
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const bool wins = (OP == 0 ? v[e] > best[c][e] : v[e] < best[c][e]) ||
                            (v[e] == best[c][e] && j < who[c][e]);
          if (wins) {
            best[c][e] = v[e];
            who[c][e] = j;
          }
        }
      }
    }

    const bool fin = act && (d.z & kLast);
    const bool heavy = fin && d.y < p.n_chunks;
    bool write = fin && !heavy;
    if (heavy) {
      const int hid = p.items[d.y].w;
      unsigned long long* pk = p.packed + int64_t(hid) * p.F;
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const uint32_t key = OP == 0 ? float_key(best[c][e]) : ~float_key(best[c][e]);
          const unsigned long long word =
              (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~who[c][e]);
          atomicMax(pk + (t * NC + c) * VEC + e, word);
        }
      __threadfence();
      const unsigned gmask = group_mask<TPR>(g);
      __syncwarp(gmask);
      int old = 0;
      if (t == 0) old = atomicAdd(p.cnt + hid, 1);
      old = __shfl_sync(gmask, old, g * TPR);
      if (old == p.hfirst[hid + 1] - p.hfirst[hid] - 1) {  // the last chunk of the node
        __threadfence();
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const unsigned long long word = atomicExch(pk + (t * NC + c) * VEC + e, 0ull);
            const uint32_t key = static_cast<uint32_t>(word >> 32);
            best[c][e] = key_float(OP == 0 ? key : ~key);
            who[c][e] = static_cast<int>(~static_cast<uint32_t>(word));
          }
        __syncwarp(gmask);
        if (t == 0) p.cnt[hid] = 0;
        write = true;
      }
    }
    if (write) {
      char* ob = static_cast<char*>(p.out) + int64_t(d.x) * RB;
      int32_t* ab = p.arg + int64_t(d.x) * p.F;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const bool none = who[c][0] == NONE;  // no in-edge at all (every element alike)
        if constexpr (sizeof(T) == 2) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = none ? 0.f : best[c][2 * q], hi = none ? 0.f : best[c][2 * q + 1];
            // exact: every value is an input bf16
            w[q] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xffff0000u);
          }
          *reinterpret_cast<uint4*>(ob + (t * NC + c) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
          *reinterpret_cast<float4*>(ob + (t * NC + c) * 16) =
              none ? make_float4(0.f, 0.f, 0.f, 0.f)
                   : make_float4(best[c][0], best[c][1], best[c][2], best[c][3]);
        }
#pragma unroll
        for (int e = 0; e < VEC; e += 4)
          *reinterpret_cast<int4*>(ab + (t * NC + c) * VEC + e) =
              none ? make_int4(-1, -1, -1, -1)
                   : make_int4(who[c][e], who[c][e + 1], who[c][e + 2], who[c][e + 3]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  ring.release(lane);
}

// dx accumulation: acc[arg[i][f]][f] += dout[i][f], 4 elements per thread.
template <typename T>
__global__ void pool_bwd_scatter_kernel(const int32_t* __restrict__ arg, const T* __restrict__ dout,
                                        float* __restrict__ acc, int64_t n4, int F) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < n4; q += stride) {
    const int4 a = reinterpret_cast<const int4*>(arg)[q];
    float g[4];
    if constexpr (sizeof(T) == 2) {
      const uint2 u = reinterpret_cast<const uint2*>(dout)[q];
      g[0] = __uint_as_float(u.x << 16);
      g[1] = __uint_as_float(u.x & 0xffff0000u);
      g[2] = __uint_as_float(u.y << 16);
      g[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
      const float4 u = reinterpret_cast<const float4*>(dout)[q];
      g[0] = u.x;
      g[1] = u.y;
      g[2] = u.z;
      g[3] = u.w;
    }
    const int f0 = int((q * 4) % F);
    const int js[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (js[e] >= 0) atomicAdd(acc + int64_t(js[e]) * F + f0 + e, g[e]);
  }
}

template <typename T>
__global__ void pool_bwd_finish_kernel(const float* __restrict__ acc, T* __restrict__ dx, int64_t n) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride) {
    if constexpr (sizeof(T) == 2) dx[e] = __float2bfloat16_rn(acc[e]);
    else dx[e] = acc[e];
  }
}

}  // namespace gattn

namespace gattn {

// Launch the pooling forward for one (dtype, row bytes): stage bytes sb
// (kStageSmall / kStageLarge) and op (0 max, 1 min) chosen at run time.
template <typename T, int RB>
gattn_status pool_dispatch(int sb, int op, const PoolParams& p, int num_sms, cudaStream_t st) {
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
  static int cache[2][2] = {{0, 0}, {0, 0}};
  const int si = sb == 4096 ? 0 : 1;
  if (sb == 4096) {
    using Sh = PoolShape<T, RB, 4096>;
    return op == 0 ? go(pool_fwd_kernel<T, RB, 4096, 0>, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[si][0])
                   : go(pool_fwd_kernel<T, RB, 4096, 1>, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[si][1]);
  }
  using Sh = PoolShape<T, RB, 8192>;
  return op == 0 ? go(pool_fwd_kernel<T, RB, 8192, 0>, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[si][0])
                 : go(pool_fwd_kernel<T, RB, 8192, 1>, Sh::THREADS, Sh::WARPS, Sh::SMEM, &cache[si][1]);
}

#define GATTN_DECLARE_POOL(TNAME, RB_)                                                    \
  gattn_status launch_pool_##TNAME##_##RB_(int sb, int op, const PoolParams& p, int num_sms, \
                                           cudaStream_t st);
#define GATTN_FOR_POOL_ROWS(X, TNAME) \
  X(TNAME, 32) X(TNAME, 64) X(TNAME, 128) X(TNAME, 256) X(TNAME, 512) X(TNAME, 1024) X(TNAME, 2048)
GATTN_FOR_POOL_ROWS(GATTN_DECLARE_POOL, f32)
GATTN_FOR_POOL_ROWS(GATTN_DECLARE_POOL, bf16)

}  // namespace gattn
