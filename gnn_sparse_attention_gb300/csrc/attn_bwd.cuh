// attn_bwd.cuh -- fused CSR attention backward (recompute from the LSE).
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", attention-based layers, backward pass:
// only a compact per-node statistic (the log-sum-exp) is cached, and the
// attention weights are recomputed on the fly; the transposed adjacency is
// cached for the backward ("Methodology", SpMM layers).
//
// With p_ij = exp(s_ij - lse_i), dp_ij = dO_i . v_j, Delta_i = dO_i . O_i
// (= sum_j p_ij dp_ij) and ds_ij = p_ij (dp_ij - Delta_i):
//   pass 1, over the CSR (a group per destination item):
//       Delta_i (written to the workspace for pass 2),
//       dot:   dQ_i = scale * sum_j ds_ij k_j
//       GATv2: dXl_i = sum_j ds_ij a . LReLU'(z_ij),  da += ds_ij LReLU(z_ij)
//   pass 2, over the cached CSC (a group per source item):
//       dot:   dK_j = scale * sum_i ds_ij q_i
//       GATv2: dXr_j = sum_i ds_ij a . LReLU'(z_ij)
//       dV_j = sum_i p_ij dO_i
// Rows arrive through the warp's cp.async ring (attn_pipe.cuh).  Heavy
// items publish partial sums and the last chunk to arrive adds them in chunk
// order.  GATv2's da is reduced warp -> block -> (last block) over the block
// partials in block order, so every result is deterministic.
#pragma once

#include "attn_pipe.cuh"

namespace gattn {

struct BwdParams {
  const int4* items;   // plan items (w = heavy id of a chunk)
  const int4* sorted;  // items by decreasing length
  int64_t n_items;
  int64_t n_chunks;    // items [0, n_chunks) are heavy chunks
  const int32_t* idx;  // pass 1: CSR sources; pass 2: CSC destinations
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const void* dO;
  const float* lse;
  float* delta;        // [N, H] workspace
  void* G1;            // pass 1: dQ;  pass 2: dK
  void* G2;            // pass 2: dV
  float* da;           // GATv2 [H*D] or null
  const float* a;
  float qmul;          // DOT: scale * log2(e)
  float scale;         // DOT: scale
  float slope;
  int H, D;
  int rows16;          // lse rows may be copied in 16-byte pieces (H % 4 == 0, lse 16-B aligned)
  int delta16;         // Delta rows may be copied in 16-byte pieces (H % 4 == 0)
  float* part;         // partials per tree slot: pass 1 [slots][HD], pass 2 [slots][2*HD]
  Tree tree;           // merge trees of the heavy items of this pass
  float* da_part;      // [gridDim.x][HD]
  int32_t* da_cnt;
  int32_t* err;        // set when a wait gives up
};

// Largest per-node fp32 row (lse or Delta): H <= RB/16 floats, padded to 16 B.
template <int RB>
struct StatBytes {
  static constexpr int value = RB / 4 < 16 ? 16 : RB / 4;
};

template <typename T, int RB>
struct CsrShape {
  using L = Lay<T, RB>;
  static constexpr int LS = StatBytes<RB>::value;
  // per item: Q, dO, O rows and the lse row; per edge: K row, V row
  static constexpr int STAGE = L::G * (3 * RB + LS) + 2 * L::B * RB;
  static constexpr int WARP_BYTES = kStages * STAGE + L::META;
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

template <typename T, int RB>
struct CscShape {
  using L = Lay<T, RB>;
  static constexpr int LS = StatBytes<RB>::value;
  // per item: K, V rows; per edge: Q row, dO row, lse row, Delta row
  static constexpr int STAGE = L::G * 2 * RB + L::B * (2 * RB + 2 * LS);
  static constexpr int WARP_BYTES = kStages * STAGE + L::META;
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

// Copy the fp32 rows src + node_r * H (r < n, node_r < 0: skip) to
// dst + r * LS, node_r taken from lane r of `nodes`.  Uniform trip count.
template <int LS>
__device__ __forceinline__ void copy_stat_rows(uint8_t* dst, const float* src, int nodes, int n,
                                               int H, bool rows16, int lane) {
  constexpr unsigned FULL = 0xffffffffu;
  const int per = rows16 ? H / 4 : H;  // pieces per row
  const int trips = (n * per + 31) / 32;
  for (int tr = 0; tr < trips; ++tr) {
    const int x = tr * 32 + lane;
    const int r = x / per, f = x % per;
    const int i = __shfl_sync(FULL, nodes, r & 31);
    if (x < n * per && i >= 0) {
      if (rows16) cp_async16(dst + r * LS + f * 16, src + int64_t(i) * H + f * 4);
      else cp_async4(dst + r * LS + f * 4, src + int64_t(i) * H + f);
    }
  }
}

// ---------------------------------------------------------------------------
// pass 1: CSR
// ---------------------------------------------------------------------------
template <typename T, int RB, int DB, int KIND>
__global__ void __launch_bounds__(CsrShape<T, RB>::THREADS) bwd_csr_kernel(const BwdParams p) {
  using L = Lay<T, RB>;
  using Sh = CsrShape<T, RB>;
  using PR = Pairs<T>;
  constexpr int NC = L::NC, TPR = L::TPR, G = L::G, SE = L::SE, B = L::B;
  constexpr int NCH = L::NCH, PP = PR::P, S = kStages, LS = Sh::LS;
  constexpr int HD = RB / (int)sizeof(T);
  constexpr int D = DB / (int)sizeof(T);  // head width
  constexpr int CPH = DB / 16;            // 16-byte chunks per head
  constexpr bool GAT = KIND == GATTN_SCORE_GATV2;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int g = lane / TPR, t = lane % TPR;
  Ring<L, Sh::STAGE> ring;
  ring.init(smem + (threadIdx.x >> 5) * Sh::WARP_BYTES, lane);
  const char* __restrict__ Qb = static_cast<const char*>(p.Q);
  const char* __restrict__ Kb = static_cast<const char*>(p.K);
  const char* __restrict__ Vb = static_cast<const char*>(p.V);
  const char* __restrict__ Ob = static_cast<const char*>(p.O);
  const char* __restrict__ dOb = static_cast<const char*>(p.dO);

  int elem[NC], head[NC];
  bool hw[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    elem[c] = (t * NC + c) * (16 / (int)sizeof(T));
    head[c] = elem[c] / D;
    hw[c] = ((t * NC + c) % CPH) == 0;
  }
  float2 av[GAT ? NC : 1][PP], dacc[GAT ? NC : 1][PP];
  if (GAT) {
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int v = 0; v < PP; ++v) {
        av[c][v] = make_float2(__ldg(p.a + elem[c] + 2 * v), __ldg(p.a + elem[c] + 2 * v + 1));
        dacc[c][v] = f2s(0.f);
      }
  }

  const int64_t warp = (int64_t(blockIdx.x) * Sh::THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * Sh::THREADS) >> 5;
  BundleCursor<G, SE> cur;
  cur.start(p.sorted, p.n_items, p.idx, warp, nwarps, ring.items, lane);

  // stage: [G][Q, dO, O rows] [G][lse row] [B][K row] [B][V row]; rows by
  // TMA bulk copies (lse rows too when they are 16-byte pieces, else 4-byte
  // cp.async).  Row r: [0,G) Q, [G,2G) dO, [2G,3G) O, [3G,4G) lse, then
  // [4G, 4G+B) K and [4G+B, 4G+2B) V.
  auto issue = [&](int s) {
    const int4* dsc = ring.desc_at(s);
    const int4 dg = lane < G ? dsc[lane] : make_int4(-1, 0, 0, 0);
    if (__shfl_sync(FULL, dg.x, 0) != -3) {
      uint8_t* st = ring.stage_at(s);
      uint64_t* bar = ring.bar_at(s);
      const int ge = (lane / SE) & 31;
      const int cn = __shfl_sync(FULL, dg.x >= 0 ? (dg.z & kCntMask) : 0, ge);
      const int jv = (lane < B && lane % SE < cn) ? ring.ix_at(s)[lane] : -1;
      const int fnode = (lane < G && dg.x >= 0 && (dg.z & kFirst)) ? dg.x : -1;
      const int nq = __popc(__ballot_sync(FULL, fnode >= 0));
      const int ne = __popc(__ballot_sync(FULL, jv >= 0));
      const uint32_t bytes = nq * (3 * RB + (p.rows16 ? 4 * p.H : 0)) + ne * 2 * RB;
      fence_proxy_async();
      if (lane == 0) mbar_expect_tx(bar, bytes);
      __syncwarp();
      if (!p.rows16) copy_stat_rows<LS>(st + G * 3 * RB, p.lse, fnode, G, p.H, false, lane);
      uint8_t* kd = st + G * (3 * RB + LS);
#pragma unroll
      for (int r0 = 0; r0 < 4 * G + 2 * B; r0 += 32) {
        const int r = r0 + lane;
        const int b = r < 4 * G + B ? r - 4 * G : r - 4 * G - B;
        const int node = __shfl_sync(FULL, fnode, (r % G) & 31);
        const int j = __shfl_sync(FULL, jv, b & 31);
        if (r < 4 * G) {
          const int gg = r % G, kind = r / G;
          if (node >= 0) {
            if (kind < 3) {
              const char* src = (kind == 0 ? Qb : (kind == 1 ? dOb : Ob)) + int64_t(node) * RB;
              bulk_g2s(st + gg * 3 * RB + kind * RB, src, RB, bar);
            } else if (p.rows16) {
              bulk_g2s(st + G * 3 * RB + gg * LS, p.lse + int64_t(node) * p.H, 4 * p.H, bar);
            }
          }
        } else if (r < 4 * G + B) {
          if (j >= 0) bulk_g2s(kd + b * RB, Kb + int64_t(j) * RB, RB, bar);
        } else if (r < 4 * G + 2 * B) {
          if (j >= 0) bulk_g2s(kd + B * RB + b * RB, Vb + int64_t(j) * RB, RB, bar);
        }
      }
    }
    cp_async_commit();
  };

  for (int s = 0; s < S; ++s) cur.generate(ring.desc_at(s), ring.ix_at(s), lane);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int s = 0; s < S - 1; ++s) {
    cur.generate(ring.desc_at(S + s), ring.ix_at(S + s), lane);
    issue(s);
  }

  float2 q[NC][PP], gq[NC][PP], dq[NC][PP];
  float lse2[NC], dlt[NC];
  for (int i = 0;; ++i) {
    cur.generate(ring.desc_at(i + 2 * S - 1), ring.ix_at(i + 2 * S - 1), lane);
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
    const bool first = act && (d.z & kFirst);

    {  // item start: q, dO, Delta = dO . O, lse (every lane joins the head reduction)
      float part[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float2 o[PP];
        if (first) {
          const uint8_t* rows = st + g * 3 * RB + (t * NC + c) * 16;
          PR::load(lds16(rows), q[c]);
          PR::load(lds16(rows + RB), gq[c]);
          PR::load(lds16(rows + 2 * RB), o);
        } else {
#pragma unroll
          for (int v = 0; v < PP; ++v) o[v] = f2s(0.f);
        }
        float2 a2 = f2s(0.f);
#pragma unroll
        for (int v = 0; v < PP; ++v) a2 = f2fma(first ? gq[c][v] : f2s(0.f), o[v], a2);
        part[c] = a2.x + a2.y;
      }
      head_totals<NC, CPH>(part);
      if (first) {
        const float* ls = reinterpret_cast<const float*>(st + G * 3 * RB + g * LS);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          dlt[c] = part[c];
          lse2[c] = ls[head[c]] * kLog2e;
          if (!GAT) {
#pragma unroll
            for (int v = 0; v < PP; ++v) q[c][v] = f2mul(q[c][v], f2s(p.qmul));
          }
#pragma unroll
          for (int v = 0; v < PP; ++v) dq[c][v] = f2s(0.f);
          // every chunk of a heavy node computes the same Delta: duplicate
          // writes store identical values
          if (hw[c]) p.delta[int64_t(d.x) * p.H + head[c]] = dlt[c];
        }
      }
    }

    const uint8_t* ks = st + G * (3 * RB + LS) + g * SE * RB;
    const uint8_t* vs = ks + B * RB;
    const int kmax = __reduce_max_sync(FULL, cnt);
#pragma unroll
    for (int k = 0; k < SE; ++k) {
      if (k >= kmax) break;
      const bool valid = k < cnt;
      float sc[NC], dp[NC];
      float2 kf[NC][PP];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int off = k * RB + (t * NC + c) * 16;
        float2 vf[PP];
        PR::load(valid ? lds16(ks + off) : make_uint4(0, 0, 0, 0), kf[c]);
        PR::load(valid ? lds16(vs + off) : make_uint4(0, 0, 0, 0), vf);
        float2 s2 = f2s(0.f), p2 = f2s(0.f);
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          p2 = f2fma(gq[c][v], vf[v], p2);
          if (!GAT) {
            s2 = f2fma(q[c][v], kf[c][v], s2);
          } else {
            const float2 z = make_float2(q[c][v].x + kf[c][v].x, q[c][v].y + kf[c][v].y);
            const float2 lr = make_float2(z.x > 0.f ? z.x : p.slope * z.x,
                                          z.y > 0.f ? z.y : p.slope * z.y);
            s2 = f2fma(av[c][v], lr, s2);
          }
        }
        sc[c] = s2.x + s2.y;
        dp[c] = p2.x + p2.y;
      }
      head_totals<NC, CPH>(sc);
      head_totals<NC, CPH>(dp);
      if (act && valid) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float pr = ex2((GAT ? sc[c] * kLog2e : sc[c]) - lse2[c]);
          const float ds = pr * (dp[c] - dlt[c]);
          if (!GAT) {
#pragma unroll
            for (int v = 0; v < PP; ++v) dq[c][v] = f2fma(f2s(ds), kf[c][v], dq[c][v]);
          } else {
#pragma unroll
            for (int v = 0; v < PP; ++v) {
              const float2 z = make_float2(q[c][v].x + kf[c][v].x, q[c][v].y + kf[c][v].y);
              const float2 sg = make_float2(z.x > 0.f ? 1.f : p.slope, z.y > 0.f ? 1.f : p.slope);
              const float2 lr = make_float2(z.x > 0.f ? z.x : p.slope * z.x,
                                            z.y > 0.f ? z.y : p.slope * z.y);
              dq[c][v] = f2fma(f2mul(f2s(ds), av[c][v]), sg, dq[c][v]);
              dacc[c][v] = f2fma(f2s(ds), lr, dacc[c][v]);
            }
          }
        }
      }
    }

    const bool fin = act && (d.z & kLast);
    const bool heavy = fin && d.y < p.n_chunks;
    bool write = fin && !heavy;
    if (heavy) {
      auto store = [&](int slot) {
        float* pb = p.part + int64_t(slot) * HD;
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; v += 2)
            *reinterpret_cast<float4*>(pb + elem[c] + 2 * v) =
                make_float4(dq[c][v].x, dq[c][v].y, dq[c][v + 1].x, dq[c][v + 1].y);
      };
      auto merge = [&](int c0, int cn) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; ++v) dq[c][v] = f2s(0.f);
        for (int kk = 0; kk < cn; kk += 4) {
          float4 f[4][NC][PP / 2];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool ok = kk + j < cn;
            const float* pc = p.part + int64_t(c0 + (ok ? kk + j : 0)) * HD;
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
              for (int v = 0; v < PP / 2; ++v)
                f[j][c][v] = ok ? __ldcg(reinterpret_cast<const float4*>(pc + elem[c] + 4 * v))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
              for (int v = 0; v < PP / 2; ++v) {
                dq[c][2 * v].x += f[j][c][v].x;
                dq[c][2 * v].y += f[j][c][v].y;
                dq[c][2 * v + 1].x += f[j][c][v].z;
                dq[c][2 * v + 1].y += f[j][c][v].w;
              }
        }
      };
      write = climb(p.tree, d.y, group_mask<TPR>(g), g * TPR, t == 0, merge, store);
    }
    if (write) {
      char* gb = static_cast<char*>(p.G1) + int64_t(d.x) * RB;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        if (!GAT) {
#pragma unroll
          for (int v = 0; v < PP; ++v) dq[c][v] = f2mul(dq[c][v], f2s(p.scale));
        }
        *reinterpret_cast<uint4*>(gb + (t * NC + c) * 16) = PR::store(dq[c]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  ring.release(lane);

  if (GAT && p.da != nullptr) {
    // warp -> block -> last block over block partials, all in fixed order
    __syncthreads();  // every warp is done with its ring: reuse shared memory
    float* s_da = reinterpret_cast<float*>(smem);  // [WARPS][HD]
    __shared__ int s_last;
#pragma unroll
    for (int o = TPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          dacc[c][v].x += __shfl_xor_sync(FULL, dacc[c][v].x, o);
          dacc[c][v].y += __shfl_xor_sync(FULL, dacc[c][v].y, o);
        }
    const int w = threadIdx.x >> 5;
    if (g == 0) {
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          s_da[w * HD + elem[c] + 2 * v] = dacc[c][v].x;
          s_da[w * HD + elem[c] + 2 * v + 1] = dacc[c][v].y;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < HD; e += Sh::THREADS) {
      float s = 0.f;
      for (int ww = 0; ww < Sh::WARPS; ++ww) s += s_da[ww * HD + e];
      p.da_part[int64_t(blockIdx.x) * HD + e] = s;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.da_cnt, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int e = threadIdx.x; e < HD; e += Sh::THREADS) {
        float s = 0.f;
        for (unsigned b = 0; b < gridDim.x; ++b) s += __ldcg(p.da_part + int64_t(b) * HD + e);
        p.da[e] = s;
      }
      if (threadIdx.x == 0) *p.da_cnt = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// pass 2: CSC
// ---------------------------------------------------------------------------
template <typename T, int RB, int DB, int KIND>
__global__ void __launch_bounds__(CscShape<T, RB>::THREADS) bwd_csc_kernel(const BwdParams p) {
  using L = Lay<T, RB>;
  using Sh = CscShape<T, RB>;
  using PR = Pairs<T>;
  constexpr int NC = L::NC, TPR = L::TPR, G = L::G, SE = L::SE, B = L::B;
  constexpr int NCH = L::NCH, PP = PR::P, S = kStages, LS = Sh::LS;
  constexpr int HD = RB / (int)sizeof(T);
  constexpr int D = DB / (int)sizeof(T);  // head width
  constexpr int CPH = DB / 16;            // 16-byte chunks per head
  constexpr bool GAT = KIND == GATTN_SCORE_GATV2;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int g = lane / TPR, t = lane % TPR;
  Ring<L, Sh::STAGE> ring;
  ring.init(smem + (threadIdx.x >> 5) * Sh::WARP_BYTES, lane);
  const char* __restrict__ Qb = static_cast<const char*>(p.Q);
  const char* __restrict__ Kb = static_cast<const char*>(p.K);
  const char* __restrict__ Vb = static_cast<const char*>(p.V);
  const char* __restrict__ dOb = static_cast<const char*>(p.dO);

  int elem[NC], head[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    elem[c] = (t * NC + c) * (16 / (int)sizeof(T));
    head[c] = elem[c] / D;
  }
  float2 av[GAT ? NC : 1][PP];
  if (GAT) {
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int v = 0; v < PP; ++v)
        av[c][v] = make_float2(__ldg(p.a + elem[c] + 2 * v), __ldg(p.a + elem[c] + 2 * v + 1));
  }

  const int64_t warp = (int64_t(blockIdx.x) * Sh::THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * Sh::THREADS) >> 5;
  BundleCursor<G, SE> cur;
  cur.start(p.sorted, p.n_items, p.idx, warp, nwarps, ring.items, lane);

  // stage: [G][K, V rows] [B][Q row] [B][dO row] [B][lse row] [B][Delta row];
  // rows by TMA bulk copies (stat rows too when they are 16-byte pieces).
  // Row r: [0,G) K, [G,2G) V, [2G, 2G+B) Q, [2G+B, 2G+2B) dO,
  // [2G+2B, 2G+3B) lse, [2G+3B, 2G+4B) Delta.
  auto issue = [&](int s) {
    const int4* dsc = ring.desc_at(s);
    const int4 dg = lane < G ? dsc[lane] : make_int4(-1, 0, 0, 0);
    if (__shfl_sync(FULL, dg.x, 0) != -3) {
      uint8_t* st = ring.stage_at(s);
      uint64_t* bar = ring.bar_at(s);
      const int ge = (lane / SE) & 31;
      const int cn = __shfl_sync(FULL, dg.x >= 0 ? (dg.z & kCntMask) : 0, ge);
      const int jv = (lane < B && lane % SE < cn) ? ring.ix_at(s)[lane] : -1;
      const int fnode = (lane < G && dg.x >= 0 && (dg.z & kFirst)) ? dg.x : -1;
      const int nq = __popc(__ballot_sync(FULL, fnode >= 0));
      const int ne = __popc(__ballot_sync(FULL, jv >= 0));
      const uint32_t bytes =
          nq * 2 * RB + ne * (2 * RB + (p.rows16 ? 4 * p.H : 0) + (p.delta16 ? 4 * p.H : 0));
      fence_proxy_async();
      if (lane == 0) mbar_expect_tx(bar, bytes);
      __syncwarp();
      uint8_t* qd = st + G * 2 * RB;
      uint8_t* gd = qd + B * RB;
      uint8_t* lsd = gd + B * RB;
      if (!p.rows16) copy_stat_rows<LS>(lsd, p.lse, jv, B, p.H, false, lane);
      if (!p.delta16) copy_stat_rows<LS>(lsd + B * LS, p.delta, jv, B, p.H, false, lane);
#pragma unroll
      for (int r0 = 0; r0 < 2 * G + 4 * B; r0 += 32) {
        const int r = r0 + lane;
        const int e = (r - 2 * G) % B;
        const int node = __shfl_sync(FULL, fnode, (r % G) & 31);
        const int i2 = __shfl_sync(FULL, jv, (e < 0 ? 0 : e) & 31);
        if (r < 2 * G) {
          if (node >= 0)
            bulk_g2s(st + (r % G) * 2 * RB + (r / G) * RB,
                     (r < G ? Kb : Vb) + int64_t(node) * RB, RB, bar);
        } else if (r < 2 * G + 4 * B && i2 >= 0) {
          const int kind = (r - 2 * G) / B;
          if (kind == 0) bulk_g2s(qd + e * RB, Qb + int64_t(i2) * RB, RB, bar);
          else if (kind == 1) bulk_g2s(gd + e * RB, dOb + int64_t(i2) * RB, RB, bar);
          else if (kind == 2 && p.rows16)
            bulk_g2s(lsd + e * LS, p.lse + int64_t(i2) * p.H, 4 * p.H, bar);
          else if (kind == 3 && p.delta16)
            bulk_g2s(lsd + B * LS + e * LS, p.delta + int64_t(i2) * p.H, 4 * p.H, bar);
        }
      }
    }
    cp_async_commit();
  };

  for (int s = 0; s < S; ++s) cur.generate(ring.desc_at(s), ring.ix_at(s), lane);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int s = 0; s < S - 1; ++s) {
    cur.generate(ring.desc_at(S + s), ring.ix_at(S + s), lane);
    issue(s);
  }

  float2 k[NC][PP], vv[NC][PP], dk[NC][PP], dv[NC][PP];
  for (int i = 0;; ++i) {
    cur.generate(ring.desc_at(i + 2 * S - 1), ring.ix_at(i + 2 * S - 1), lane);
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
      for (int c = 0; c < NC; ++c) {
        const uint8_t* rows = st + g * 2 * RB + (t * NC + c) * 16;
        PR::load(lds16(rows), k[c]);
        PR::load(lds16(rows + RB), vv[c]);
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          if (!GAT) k[c][v] = f2mul(k[c][v], f2s(p.qmul));
          dk[c][v] = dv[c][v] = f2s(0.f);
        }
      }
    }

    const uint8_t* qs = st + G * 2 * RB + g * SE * RB;
    const uint8_t* gs = qs + B * RB;
    const float* lss = reinterpret_cast<const float*>(st + G * 2 * RB + 2 * B * RB) + g * SE * (LS / 4);
    const float* dls = lss + B * (LS / 4);
    const int kmax = __reduce_max_sync(FULL, cnt);
#pragma unroll
    for (int e = 0; e < SE; ++e) {
      if (e >= kmax) break;
      const bool valid = e < cnt;
      float sc[NC], dp[NC];
      float2 qf[NC][PP], gf[NC][PP];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int off = e * RB + (t * NC + c) * 16;
        PR::load(valid ? lds16(qs + off) : make_uint4(0, 0, 0, 0), qf[c]);
        PR::load(valid ? lds16(gs + off) : make_uint4(0, 0, 0, 0), gf[c]);
        float2 s2 = f2s(0.f), p2 = f2s(0.f);
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          p2 = f2fma(gf[c][v], vv[c][v], p2);
          if (!GAT) {
            s2 = f2fma(qf[c][v], k[c][v], s2);
          } else {
            const float2 z = make_float2(qf[c][v].x + k[c][v].x, qf[c][v].y + k[c][v].y);
            const float2 lr = make_float2(z.x > 0.f ? z.x : p.slope * z.x,
                                          z.y > 0.f ? z.y : p.slope * z.y);
            s2 = f2fma(av[c][v], lr, s2);
          }
        }
        sc[c] = s2.x + s2.y;
        dp[c] = p2.x + p2.y;
      }
      head_totals<NC, CPH>(sc);
      head_totals<NC, CPH>(dp);
      if (act && valid) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float ls = lss[e * (LS / 4) + head[c]];
          const float dl = dls[e * (LS / 4) + head[c]];
          const float pr = ex2((GAT ? sc[c] * kLog2e : sc[c]) - ls * kLog2e);
          const float ds = pr * (dp[c] - dl);
#pragma unroll
          for (int v = 0; v < PP; ++v) dv[c][v] = f2fma(f2s(pr), gf[c][v], dv[c][v]);
          if (!GAT) {
#pragma unroll
            for (int v = 0; v < PP; ++v) dk[c][v] = f2fma(f2s(ds), qf[c][v], dk[c][v]);
          } else {
#pragma unroll
            for (int v = 0; v < PP; ++v) {
              const float2 z = make_float2(qf[c][v].x + k[c][v].x, qf[c][v].y + k[c][v].y);
              const float2 sg = make_float2(z.x > 0.f ? 1.f : p.slope, z.y > 0.f ? 1.f : p.slope);
              dk[c][v] = f2fma(f2mul(f2s(ds), av[c][v]), sg, dk[c][v]);
            }
          }
        }
      }
    }

    const bool fin = act && (d.z & kLast);
    const bool heavy = fin && d.y < p.n_chunks;
    bool write = fin && !heavy;
    if (heavy) {
      constexpr int HD = RB / (int)sizeof(T);
      auto store = [&](int slot) {
        float* pb = p.part + int64_t(slot) * (2 * HD);
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; v += 2) {
            *reinterpret_cast<float4*>(pb + elem[c] + 2 * v) =
                make_float4(dk[c][v].x, dk[c][v].y, dk[c][v + 1].x, dk[c][v + 1].y);
            *reinterpret_cast<float4*>(pb + HD + elem[c] + 2 * v) =
                make_float4(dv[c][v].x, dv[c][v].y, dv[c][v + 1].x, dv[c][v + 1].y);
          }
      };
      auto merge = [&](int c0, int cn) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; ++v) dk[c][v] = dv[c][v] = f2s(0.f);
        for (int kk = 0; kk < cn; kk += 2) {
          float4 f[2][NC][PP / 2], h[2][NC][PP / 2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const bool ok = kk + j < cn;
            const float* pc = p.part + int64_t(c0 + (ok ? kk + j : 0)) * (2 * HD);
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
              for (int v = 0; v < PP / 2; ++v) {
                f[j][c][v] = ok ? __ldcg(reinterpret_cast<const float4*>(pc + elem[c] + 4 * v))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                h[j][c][v] = ok ? __ldcg(reinterpret_cast<const float4*>(pc + HD + elem[c] + 4 * v))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
              }
          }
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
              for (int v = 0; v < PP / 2; ++v) {
                dk[c][2 * v].x += f[j][c][v].x;
                dk[c][2 * v].y += f[j][c][v].y;
                dk[c][2 * v + 1].x += f[j][c][v].z;
                dk[c][2 * v + 1].y += f[j][c][v].w;
                dv[c][2 * v].x += h[j][c][v].x;
                dv[c][2 * v].y += h[j][c][v].y;
                dv[c][2 * v + 1].x += h[j][c][v].z;
                dv[c][2 * v + 1].y += h[j][c][v].w;
              }
        }
      };
      write = climb(p.tree, d.y, group_mask<TPR>(g), g * TPR, t == 0, merge, store);
    }
    if (write) {
      char* kb = static_cast<char*>(p.G1) + int64_t(d.x) * RB;
      char* vb = static_cast<char*>(p.G2) + int64_t(d.x) * RB;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        if (!GAT) {
#pragma unroll
          for (int v = 0; v < PP; ++v) dk[c][v] = f2mul(dk[c][v], f2s(p.scale));
        }
        *reinterpret_cast<uint4*>(kb + (t * NC + c) * 16) = PR::store(dk[c]);
        *reinterpret_cast<uint4*>(vb + (t * NC + c) * 16) = PR::store(dv[c]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  ring.release(lane);
}

}  // namespace gattn
