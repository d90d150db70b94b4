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
//   pass 1, over the CSR (warp per destination item):
//       Delta_i (written to the workspace for pass 2),
//       dot:   dQ_i = scale * sum_j ds_ij k_j
//       GATv2: dXl_i = sum_j ds_ij a . LReLU'(z_ij),  da += ds_ij LReLU(z_ij)
//   pass 2, over the cached CSC (warp per source item):
//       dot:   dK_j = scale * sum_i ds_ij q_i
//       GATv2: dXr_j = sum_i ds_ij a . LReLU'(z_ij)
//       dV_j = sum_i p_ij dO_i
// Heavy items publish partial sums and the last chunk to arrive adds them
// in chunk order.  GATv2's da is reduced warp -> block -> (last block) over
// the block partials in block order, so every result is deterministic.
#pragma once

#include "gattn_internal.cuh"

namespace gattn {

struct BwdParams {
  const int4* items;
  int64_t n_items;
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
  float* part;         // chunk partials: pass 1 [n_chunks][HD], pass 2 [n_chunks][2*HD]
  int32_t* cnt;
  const int32_t* hfirst;
  float* da_part;      // [gridDim.x][HD]
  int32_t* da_cnt;
};

template <int VEC>
__device__ __forceinline__ void load_f32x(const float* p, float* x) {
#pragma unroll
  for (int v = 0; v < VEC; v += 4) {
    const float4 f = __ldcg(reinterpret_cast<const float4*>(p + v));
    x[v] = f.x;
    x[v + 1] = f.y;
    x[v + 2] = f.z;
    x[v + 3] = f.w;
  }
}
template <int VEC>
__device__ __forceinline__ void store_f32x(float* p, const float* x) {
#pragma unroll
  for (int v = 0; v < VEC; v += 4)
    *reinterpret_cast<float4*>(p + v) = make_float4(x[v], x[v + 1], x[v + 2], x[v + 3]);
}

// ---------------------------------------------------------------------------
// pass 1: CSR
// ---------------------------------------------------------------------------
template <typename T, int RB, int KIND>
__global__ void __launch_bounds__(kThreads) bwd_csr_kernel(const BwdParams p) {
  using L = Layout<T, RB>;
  constexpr int VEC = L::VEC, CPL = L::CPL, LPR = L::LPR, EPW = L::EPW, U = L::U, B = L::B;
  constexpr int HD = RB / (int)sizeof(T);
  constexpr bool GAT = KIND == GATTN_SCORE_GATV2;
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int slot = lane / LPR;
  const int rl = lane % LPR;
  const int lph = p.D / VEC;
  const char* __restrict__ Qb = static_cast<const char*>(p.Q);
  const char* __restrict__ Kb = static_cast<const char*>(p.K);
  const char* __restrict__ Vb = static_cast<const char*>(p.V);
  const char* __restrict__ Ob = static_cast<const char*>(p.O);
  const char* __restrict__ dOb = static_cast<const char*>(p.dO);

  int elem[CPL], head[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    elem[c] = (c * LPR + rl) * VEC;
    head[c] = elem[c] / p.D;
  }
  float av[GAT ? CPL : 1][VEC];
  float dacc[GAT ? CPL : 1][VEC];
  if (GAT) {
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        av[c][v] = __ldg(p.a + elem[c] + v);
        dacc[c][v] = 0.f;
      }
  }

  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  for (int64_t it = warp; it < p.n_items; it += nwarps) {
    const int4 item = p.items[it];
    const int node = item.x, e0 = item.y, e1 = item.z, hid = item.w;
    const int64_t nrow = int64_t(node) * RB;

    float q[CPL][VEC], g[CPL][VEC], lse2[CPL], dlt[CPL], dq[CPL][VEC];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      float o[VEC];
      Cvt<T>::to_f32(ldg16(Qb + nrow + elem[c] * sizeof(T)), q[c]);
      Cvt<T>::to_f32(ldg16(dOb + nrow + elem[c] * sizeof(T)), g[c]);
      Cvt<T>::to_f32(ldg16(Ob + nrow + elem[c] * sizeof(T)), o);
      float t = 0.f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) t = fmaf(g[c][v], o[v], t);
      dlt[c] = head_sum(t, lph);
      lse2[c] = __ldg(p.lse + int64_t(node) * p.H + head[c]) * kLog2e;
      if (!GAT) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) q[c][v] *= p.qmul;
      }
#pragma unroll
      for (int v = 0; v < VEC; ++v) dq[c][v] = 0.f;
    }
    if ((hid < 0 || it == p.hfirst[hid]) && slot == 0) {
#pragma unroll
      for (int c = 0; c < CPL; ++c)
        if (rl % lph == 0) p.delta[int64_t(node) * p.H + head[c]] = dlt[c];
    }

    for (int eb = e0; eb < e1; eb += 32) {
      const int nb = min(32, e1 - eb);
      const int myj = lane < nb ? __ldg(p.idx + eb + lane) : 0;
      for (int sb = 0; sb < nb; sb += B) {
        uint4 kr[U][CPL], vr[U][CPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int eo = sb + u * EPW + slot;
          const int j = __shfl_sync(FULL, myj, eo);
          if (eo < nb) {
            const int64_t row = int64_t(j) * RB;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              kr[u][c] = ldg16(Kb + row + elem[c] * sizeof(T));
              vr[u][c] = ldg16(Vb + row + elem[c] * sizeof(T));
            }
          } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) kr[u][c] = vr[u][c] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool valid = sb + u * EPW + slot < nb;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float k[VEC], vv[VEC];
            Cvt<T>::to_f32(kr[u][c], k);
            Cvt<T>::to_f32(vr[u][c], vv);
            float t = 0.f, dp = 0.f;
#pragma unroll
            for (int v = 0; v < VEC; ++v) dp = fmaf(g[c][v], vv[v], dp);
            if (!GAT) {
#pragma unroll
              for (int v = 0; v < VEC; ++v) t = fmaf(q[c][v], k[v], t);
              t = head_sum(t, lph);
            } else {
#pragma unroll
              for (int v = 0; v < VEC; ++v) {
                const float z = q[c][v] + k[v];
                t = fmaf(av[c][v], z > 0.f ? z : p.slope * z, t);
              }
              t = head_sum(t, lph) * kLog2e;
            }
            dp = head_sum(dp, lph);
            const float pr = valid ? ex2(t - lse2[c]) : 0.f;
            const float ds = pr * (dp - dlt[c]);
            if (!GAT) {
#pragma unroll
              for (int v = 0; v < VEC; ++v) dq[c][v] = fmaf(ds, k[v], dq[c][v]);
            } else {
#pragma unroll
              for (int v = 0; v < VEC; ++v) {
                const float z = q[c][v] + k[v];
                const bool pos = z > 0.f;
                dq[c][v] = fmaf(ds * av[c][v], pos ? 1.f : p.slope, dq[c][v]);
                dacc[c][v] = fmaf(ds, pos ? z : p.slope * z, dacc[c][v]);
              }
            }
          }
        }
      }
    }

#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < VEC; ++v) dq[c][v] += __shfl_xor_sync(FULL, dq[c][v], o);

    bool write_final = hid < 0;
    if (!write_final) {
      float* pb = p.part + it * int64_t(HD);
      if (slot == 0) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) store_f32x<VEC>(pb + elem[c], dq[c]);
      }
      __threadfence();
      __syncwarp();
      int old = 0;
      if (lane == 0) old = atomicAdd(p.cnt + hid, 1);
      old = __shfl_sync(FULL, old, 0);
      const int first = p.hfirst[hid];
      const int n = p.hfirst[hid + 1] - first;
      if (old == n - 1) {
        __threadfence();
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
          for (int v = 0; v < VEC; ++v) dq[c][v] = 0.f;
        for (int k = slot; k < n; k += EPW) {
          const float* pc = p.part + int64_t(first + k) * HD;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float x[VEC];
            load_f32x<VEC>(pc + elem[c], x);
#pragma unroll
            for (int v = 0; v < VEC; ++v) dq[c][v] += x[v];
          }
        }
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
          for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int v = 0; v < VEC; ++v) dq[c][v] += __shfl_xor_sync(FULL, dq[c][v], o);
        if (lane == 0) p.cnt[hid] = 0;
        write_final = true;
      }
    }
    if (write_final && slot == 0) {
      char* gb = static_cast<char*>(p.G1) + nrow;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        if (!GAT) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) dq[c][v] *= p.scale;
        }
        *reinterpret_cast<uint4*>(gb + elem[c] * sizeof(T)) = Cvt<T>::from_f32(dq[c]);
      }
    }
  }

  if (GAT && p.da != nullptr) {
    // warp -> block -> last block over block partials, all in fixed order
    __shared__ float s_da[kWarpsPerBlock][HD];
    __shared__ int s_last;
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < VEC; ++v) dacc[c][v] += __shfl_xor_sync(FULL, dacc[c][v], o);
    const int w = threadIdx.x >> 5;
    if (slot == 0) {
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < VEC; ++v) s_da[w][elem[c] + v] = dacc[c][v];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < HD; e += kThreads) {
      float t = 0.f;
      for (int ww = 0; ww < kWarpsPerBlock; ++ww) t += s_da[ww][e];
      p.da_part[int64_t(blockIdx.x) * HD + e] = t;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.da_cnt, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int e = threadIdx.x; e < HD; e += kThreads) {
        float t = 0.f;
        for (unsigned b = 0; b < gridDim.x; ++b) t += __ldcg(p.da_part + int64_t(b) * HD + e);
        p.da[e] = t;
      }
      if (threadIdx.x == 0) *p.da_cnt = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// pass 2: CSC
// ---------------------------------------------------------------------------
template <typename T, int RB, int KIND>
__global__ void __launch_bounds__(kThreads) bwd_csc_kernel(const BwdParams p) {
  using L = Layout<T, RB>;
  constexpr int VEC = L::VEC, CPL = L::CPL, LPR = L::LPR, EPW = L::EPW, U = L::U, B = L::B;
  constexpr int HD = RB / (int)sizeof(T);
  constexpr bool GAT = KIND == GATTN_SCORE_GATV2;
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int slot = lane / LPR;
  const int rl = lane % LPR;
  const int lph = p.D / VEC;
  const char* __restrict__ Qb = static_cast<const char*>(p.Q);
  const char* __restrict__ Kb = static_cast<const char*>(p.K);
  const char* __restrict__ Vb = static_cast<const char*>(p.V);
  const char* __restrict__ dOb = static_cast<const char*>(p.dO);

  int elem[CPL], head[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    elem[c] = (c * LPR + rl) * VEC;
    head[c] = elem[c] / p.D;
  }
  float av[GAT ? CPL : 1][VEC];
  if (GAT) {
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int v = 0; v < VEC; ++v) av[c][v] = __ldg(p.a + elem[c] + v);
  }

  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  for (int64_t it = warp; it < p.n_items; it += nwarps) {
    const int4 item = p.items[it];
    const int src = item.x, e0 = item.y, e1 = item.z, hid = item.w;
    const int64_t srow = int64_t(src) * RB;

    float k[CPL][VEC], vv[CPL][VEC], dk[CPL][VEC], dv[CPL][VEC];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      Cvt<T>::to_f32(ldg16(Kb + srow + elem[c] * sizeof(T)), k[c]);
      Cvt<T>::to_f32(ldg16(Vb + srow + elem[c] * sizeof(T)), vv[c]);
      if (!GAT) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) k[c][v] *= p.qmul;
      }
#pragma unroll
      for (int v = 0; v < VEC; ++v) dk[c][v] = dv[c][v] = 0.f;
    }

    for (int eb = e0; eb < e1; eb += 32) {
      const int nb = min(32, e1 - eb);
      const int myi = lane < nb ? __ldg(p.idx + eb + lane) : 0;
      for (int sb = 0; sb < nb; sb += B) {
        uint4 qr[U][CPL], gr[U][CPL];
        float ls[U][CPL], dl[U][CPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int eo = sb + u * EPW + slot;
          const int i = __shfl_sync(FULL, myi, eo);
          if (eo < nb) {
            const int64_t row = int64_t(i) * RB;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              qr[u][c] = ldg16(Qb + row + elem[c] * sizeof(T));
              gr[u][c] = ldg16(dOb + row + elem[c] * sizeof(T));
              ls[u][c] = __ldg(p.lse + int64_t(i) * p.H + head[c]);
              dl[u][c] = __ldcg(p.delta + int64_t(i) * p.H + head[c]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              qr[u][c] = gr[u][c] = make_uint4(0, 0, 0, 0);
              ls[u][c] = dl[u][c] = 0.f;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool valid = sb + u * EPW + slot < nb;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float q[VEC], g[VEC];
            Cvt<T>::to_f32(qr[u][c], q);
            Cvt<T>::to_f32(gr[u][c], g);
            float t = 0.f, dp = 0.f;
#pragma unroll
            for (int v = 0; v < VEC; ++v) dp = fmaf(g[v], vv[c][v], dp);
            if (!GAT) {
#pragma unroll
              for (int v = 0; v < VEC; ++v) t = fmaf(q[v], k[c][v], t);
              t = head_sum(t, lph);
            } else {
#pragma unroll
              for (int v = 0; v < VEC; ++v) {
                const float z = q[v] + k[c][v];
                t = fmaf(av[c][v], z > 0.f ? z : p.slope * z, t);
              }
              t = head_sum(t, lph) * kLog2e;
            }
            dp = head_sum(dp, lph);
            const float pr = valid ? ex2(t - ls[u][c] * kLog2e) : 0.f;
            const float ds = pr * (dp - dl[u][c]);
#pragma unroll
            for (int v = 0; v < VEC; ++v) dv[c][v] = fmaf(pr, g[v], dv[c][v]);
            if (!GAT) {
#pragma unroll
              for (int v = 0; v < VEC; ++v) dk[c][v] = fmaf(ds, q[v], dk[c][v]);
            } else {
#pragma unroll
              for (int v = 0; v < VEC; ++v) {
                const float z = q[v] + k[c][v];
                dk[c][v] = fmaf(ds * av[c][v], z > 0.f ? 1.f : p.slope, dk[c][v]);
              }
            }
          }
        }
      }
    }

#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          dk[c][v] += __shfl_xor_sync(FULL, dk[c][v], o);
          dv[c][v] += __shfl_xor_sync(FULL, dv[c][v], o);
        }

    bool write_final = hid < 0;
    if (!write_final) {
      float* pb = p.part + it * int64_t(2 * HD);
      if (slot == 0) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          store_f32x<VEC>(pb + elem[c], dk[c]);
          store_f32x<VEC>(pb + HD + elem[c], dv[c]);
        }
      }
      __threadfence();
      __syncwarp();
      int old = 0;
      if (lane == 0) old = atomicAdd(p.cnt + hid, 1);
      old = __shfl_sync(FULL, old, 0);
      const int first = p.hfirst[hid];
      const int n = p.hfirst[hid + 1] - first;
      if (old == n - 1) {
        __threadfence();
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
          for (int v = 0; v < VEC; ++v) dk[c][v] = dv[c][v] = 0.f;
        for (int kk = slot; kk < n; kk += EPW) {
          const float* pc = p.part + int64_t(first + kk) * (2 * HD);
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float x[VEC], y[VEC];
            load_f32x<VEC>(pc + elem[c], x);
            load_f32x<VEC>(pc + HD + elem[c], y);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              dk[c][v] += x[v];
              dv[c][v] += y[v];
            }
          }
        }
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
          for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              dk[c][v] += __shfl_xor_sync(FULL, dk[c][v], o);
              dv[c][v] += __shfl_xor_sync(FULL, dv[c][v], o);
            }
        if (lane == 0) p.cnt[hid] = 0;
        write_final = true;
      }
    }
    if (write_final && slot == 0) {
      char* kb = static_cast<char*>(p.G1) + srow;
      char* vb = static_cast<char*>(p.G2) + srow;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        if (!GAT) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) dk[c][v] *= p.scale;
        }
        *reinterpret_cast<uint4*>(kb + elem[c] * sizeof(T)) = Cvt<T>::from_f32(dk[c]);
        *reinterpret_cast<uint4*>(vb + elem[c] * sizeof(T)) = Cvt<T>::from_f32(dv[c]);
      }
    }
  }
}

}  // namespace gattn
