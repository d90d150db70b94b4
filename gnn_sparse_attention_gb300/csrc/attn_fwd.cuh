// attn_fwd.cuh -- fused CSR attention forward.
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", attention-based layers: scores, softmax
// normalisation and value aggregation are fused into one streaming pass over
// each destination's in-neighbours; an online softmax keeps the running
// statistics in registers and only a per-node log-sum-exp is written.
//
// One warp owns one work item: a light destination (all of its edges) or one
// edge chunk of a heavy destination.  Per 32 edges the warp loads the source
// ids with one coalesced read and broadcasts them by shuffle; each slot of
// LPR lanes gathers one K row and one V row per step with 16-byte loads, U
// steps in flight before the online-softmax update.  Scores live in base-2
// units (q or a pre-multiplied by log2 e) so every exponential is one ex2.
// At the end the slots' (m, l, acc) states merge by butterfly shuffles.
//
// Heavy destinations: each chunk writes its unnormalised (acc, m, l) triple
// to the workspace, fences, and bumps the node's counter; the warp that
// arrives last merges all chunks in chunk order (a deterministic result) and
// resets the counter.  No warp ever waits on another.
#pragma once

#include "gattn_internal.cuh"

namespace gattn {

struct FwdParams {
  const int4* items;
  int64_t n_items;
  const int32_t* indices;
  const void* Q;
  const void* K;
  const void* V;
  void* out;
  float* lse;
  const float* a;  // GATv2 [H*D]
  float qmul;      // DOT: scale * log2(e)
  float slope;     // GATv2 LeakyReLU slope
  int H, D;
  float* part;     // [n_chunks][pstride]: acc[HD], m[H], l[H]
  int pstride;
  int32_t* cnt;    // [n_heavy]
  const int32_t* hfirst;
};

// (m, l, acc) <- combine((m, l, acc), (mo, lo, acco)), base-2 exponents.
template <int VEC>
__device__ __forceinline__ void softmax_combine(float& m, float& l, float* acc, float mo, float lo,
                                                const float* acco) {
  const float mn = fmaxf(m, mo);
  const float base = mn == neg_inf() ? 0.f : mn;
  const float c1 = ex2(m - base), c2 = ex2(mo - base);
  l = l * c1 + lo * c2;
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = acc[v] * c1 + acco[v] * c2;
  m = mn;
}

template <typename T, int RB, int KIND>
__global__ void __launch_bounds__(kThreads) fwd_kernel(const FwdParams p) {
  using L = Layout<T, RB>;
  constexpr int VEC = L::VEC, CPL = L::CPL, LPR = L::LPR, EPW = L::EPW, U = L::U, B = L::B;
  constexpr int HD = RB / (int)sizeof(T);
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int slot = lane / LPR;
  const int rl = lane % LPR;
  const int lph = p.D / VEC;
  const char* __restrict__ Qb = static_cast<const char*>(p.Q);
  const char* __restrict__ Kb = static_cast<const char*>(p.K);
  const char* __restrict__ Vb = static_cast<const char*>(p.V);

  int elem[CPL], head[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    elem[c] = (c * LPR + rl) * VEC;
    head[c] = elem[c] / p.D;
  }
  float av[KIND == GATTN_SCORE_GATV2 ? CPL : 1][VEC];
  if (KIND == GATTN_SCORE_GATV2) {
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int v = 0; v < VEC; ++v) av[c][v] = __ldg(p.a + elem[c] + v);
  }

  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  for (int64_t it = warp; it < p.n_items; it += nwarps) {
    const int4 item = p.items[it];
    const int node = item.x, e0 = item.y, e1 = item.z, hid = item.w;

    float q[CPL][VEC];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      Cvt<T>::to_f32(ldg16(Qb + int64_t(node) * RB + elem[c] * sizeof(T)), q[c]);
      if (KIND == GATTN_SCORE_DOT) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) q[c][v] *= p.qmul;
      }
    }
    float m[CPL], l[CPL], acc[CPL][VEC];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      m[c] = neg_inf();
      l[c] = 0.f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[c][v] = 0.f;
    }

    for (int eb = e0; eb < e1; eb += 32) {
      const int nb = min(32, e1 - eb);
      const int myj = lane < nb ? __ldg(p.indices + eb + lane) : 0;
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
        float s[U][CPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float k[VEC];
            Cvt<T>::to_f32(kr[u][c], k);
            float t = 0.f;
            if (KIND == GATTN_SCORE_DOT) {
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
            s[u][c] = (sb + u * EPW + slot < nb) ? t : neg_inf();
          }
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float mx = m[c];
#pragma unroll
          for (int u = 0; u < U; ++u) mx = fmaxf(mx, s[u][c]);
          const float base = mx == neg_inf() ? 0.f : mx;
          const float corr = ex2(m[c] - base);
          l[c] *= corr;
#pragma unroll
          for (int v = 0; v < VEC; ++v) acc[c][v] *= corr;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const float pu = ex2(s[u][c] - base);
            l[c] += pu;
            float vv[VEC];
            Cvt<T>::to_f32(vr[u][c], vv);
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[c][v] = fmaf(pu, vv[v], acc[c][v]);
          }
          m[c] = mx;
        }
      }
    }

    // merge the warp's slots
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float acco[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) acco[v] = __shfl_xor_sync(FULL, acc[c][v], o);
        const float mo = __shfl_xor_sync(FULL, m[c], o);
        const float lo = __shfl_xor_sync(FULL, l[c], o);
        softmax_combine<VEC>(m[c], l[c], acc[c], mo, lo, acco);
      }
    }

    bool write_final = hid < 0;
    if (!write_final) {
      // heavy chunk: publish the partial, the last chunk to arrive merges
      float* pb = p.part + it * int64_t(p.pstride);
      if (slot == 0) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float4* dst = reinterpret_cast<float4*>(pb + elem[c]);
#pragma unroll
          for (int v = 0; v < VEC; v += 4)
            dst[v / 4] = make_float4(acc[c][v], acc[c][v + 1], acc[c][v + 2], acc[c][v + 3]);
          if (rl % lph == 0) {
            pb[HD + head[c]] = m[c];
            pb[HD + p.H + head[c]] = l[c];
          }
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
        for (int c = 0; c < CPL; ++c) {
          m[c] = neg_inf();
          l[c] = 0.f;
#pragma unroll
          for (int v = 0; v < VEC; ++v) acc[c][v] = 0.f;
        }
        for (int k = slot; k < n; k += EPW) {
          const float* pc = p.part + int64_t(first + k) * p.pstride;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float acco[VEC];
#pragma unroll
            for (int v = 0; v < VEC; v += 4) {
              const float4 f = __ldcg(reinterpret_cast<const float4*>(pc + elem[c] + v));
              acco[v] = f.x;
              acco[v + 1] = f.y;
              acco[v + 2] = f.z;
              acco[v + 3] = f.w;
            }
            const float mo = __ldcg(pc + HD + head[c]);
            const float lo = __ldcg(pc + HD + p.H + head[c]);
            softmax_combine<VEC>(m[c], l[c], acc[c], mo, lo, acco);
          }
        }
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float acco[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) acco[v] = __shfl_xor_sync(FULL, acc[c][v], o);
            const float mo = __shfl_xor_sync(FULL, m[c], o);
            const float lo = __shfl_xor_sync(FULL, l[c], o);
            softmax_combine<VEC>(m[c], l[c], acc[c], mo, lo, acco);
          }
        }
        if (lane == 0) p.cnt[hid] = 0;
        write_final = true;
      }
    }
    if (write_final && slot == 0) {
      char* ob = static_cast<char*>(p.out) + int64_t(node) * RB;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float inv = l[c] > 0.f ? 1.f / l[c] : 0.f;
        float o[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = acc[c][v] * inv;
        *reinterpret_cast<uint4*>(ob + elem[c] * sizeof(T)) = Cvt<T>::from_f32(o);
        if (rl % lph == 0)
          p.lse[int64_t(node) * p.H + head[c]] = l[c] > 0.f ? (m[c] + lg2(l[c])) * kLn2 : neg_inf();
      }
    }
  }
}

}  // namespace gattn
