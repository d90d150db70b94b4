// attn_fwd.cuh -- fused CSR attention forward.
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", attention-based layers: scores, softmax
// normalisation and value aggregation are fused into one streaming pass over
// each destination's in-neighbours; an online softmax keeps the running
// statistics in registers and only a per-node log-sum-exp is written.
//
// Each group of TPR lanes owns one work item (a light destination with all
// of its edges, or one edge chunk of a heavy destination) and each lane a
// 32-byte slice of the rows (see attn_pipe.cuh).  The item's Q row and the
// K and V rows of its in-neighbours arrive through the warp's cp.async ring.
// Per stage a lane scores its SE edges (packed fp32 FMAs), takes one running
// max over them, rescales once and accumulates the values.  Scores live in
// base-2 units (q or a pre-multiplied by log2 e), so every exponential is one
// ex2.
//
// Heavy destinations: each chunk writes its unnormalised (acc, m, l) triple
// to the workspace, fences, and bumps the node's counter; the group that
// arrives last merges all chunks in chunk order (a deterministic result) and
// resets the counter.  No lane ever waits on another.
#pragma once

#include "attn_pipe.cuh"

namespace gattn {

struct FwdParams {
  CUtensorMap mq, mk, mv;  // row-gather maps of Q, K, V (tma.cuh)
  const int4* items;   // plan items (w = heavy id of a chunk)
  const int4* sorted;  // items by decreasing length
  int64_t n_items;
  int64_t n_chunks;    // items [0, n_chunks) are heavy chunks
  int N;               // rows of Q, K, V; row index N is the zero-filled pad row
  const int32_t* indices;
  const void* Q;
  const void* K;
  const void* V;
  void* out;
  float* lse;
  const float* a;      // GATv2 [H*D]
  float qmul;          // DOT: scale * log2(e)
  float slope;         // GATv2 LeakyReLU slope
  int H, D;
  float* part;         // [n_chunks + n_inner][pstride]: acc[HD], m[H], l[H]
  int pstride;
  Tree tree;           // merge trees of the heavy destinations
  int32_t* err;        // set when a wait gives up
  int fail_first_wait; // nonzero: every warp's first wait expires at once (failure-path test)
};

template <typename T, int RB, int SB>
struct FwdShape {
  using L = Lay<T, RB, SB>;
  // Item rows inline (attn_pipe.cuh, BundleCursor) where a stage holds whole
  // 4-row sets and at least 4 edges per item: a starting item's Q row takes
  // the K-row slot of its group's last edge position.  Otherwise (short
  // stages, where one edge position less per item would cost a stage in
  // most items) Q rows have a region of their own (IR slots).
  static constexpr int RES = (L::G >= 4 && L::SE >= 4) ? 1 : 0;
  static constexpr int IRS = RES ? 0 : L::IR;
  // [IRS Q rows] then B K rows and B V rows
  static constexpr int STAGE = RB * (IRS + 2 * L::B);
  static constexpr int WARP_BYTES = align128(kStages * STAGE + L::META);
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int MINB = WarpsFor<WARP_BYTES>::minb;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

template <typename T, int RB, int DB, int KIND, int SB>
__global__ void __launch_bounds__(FwdShape<T, RB, SB>::THREADS, min_blocks<FwdShape<T, RB, SB>::WARP_BYTES, RB, SB>(KIND)) fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = Lay<T, RB, SB>;
  using Sh = FwdShape<T, RB, SB>;
  using PR = Pairs<T>;
  constexpr int NC = L::NC, TPR = L::TPR, G = L::G, SE = L::SE, B = L::B;
  constexpr int PP = PR::P, S = kStages;
  constexpr int HD = RB / (int)sizeof(T);
  constexpr int D = DB / (int)sizeof(T);  // head width
  constexpr int CPH = DB / 16;            // 16-byte chunks per head
  using LH = LaneHeads<NC, CPH>;
  constexpr int HL = LH::N;               // heads of this lane
  constexpr bool GAT = KIND == GATTN_SCORE_GATV2;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int g = lane / TPR, t = lane % TPR;
  Ring<L, Sh::STAGE> ring;
  ring.init(smem + (threadIdx.x >> 5) * Sh::WARP_BYTES, lane);

  // this lane's chunks: global chunk t*NC + c of the row, its head, and
  // whether the lane writes that head's per-head values
  int elem[NC], head[NC];
  bool hw[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    elem[c] = (t * NC + c) * (16 / (int)sizeof(T));
    head[c] = elem[c] / D;
    hw[c] = ((t * NC + c) % CPH) == 0;
  }
  // GATv2: a . LReLU(z) = (a c1) . z + (a c2) . |z| (attn_pipe.cuh)
  float2 ac1[GAT ? NC : 1][PP], ac2[GAT ? NC : 1][PP];
  if (GAT) {
    const float c1 = 0.5f * (1.f + p.slope), c2 = 0.5f * (1.f - p.slope);
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int v = 0; v < PP; ++v) {
        const float2 a2 = make_float2(__ldg(p.a + elem[c] + 2 * v), __ldg(p.a + elem[c] + 2 * v + 1));
        ac1[c][v] = f2mul(a2, f2s(c1));
        ac2[c][v] = f2mul(a2, f2s(c2));
      }
  }

  const int64_t warp = (int64_t(blockIdx.x) * Sh::THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * Sh::THREADS) >> 5;
  using Cur = BundleCursor<G, SE, Sh::RES>;
  Cur cur;
  cur.start(p.sorted, p.n_items, p.indices, p.N, warp, nwarps, ring.items, lane);

  // rows of stage s into its ring slot by TMA gathers issued from lane 0:
  // Q rows of the items that start here (only the 4-row sets that hold one),
  // then the K rows and the V rows of the stage's edges; unused slots gather
  // the zero-filled pad row N.  With inline item rows, a stage that starts a
  // bundle gathers the Q rows into the K slots of the last edge position and
  // skips that position's V slots.  Bytes are counted on the slot's barrier.
    // rows of stage s into its ring slot by TMA gathers issued from lane 0:
  // Q rows of the items that start here (only the 4-row sets that hold one),
  // then the K rows and the V rows of the stage's edges; unused slots gather
  // the zero-filled pad row N.  With inline item rows, a stage that starts a
  // bundle gathers the Q rows into the K slots of the last edge position and
  // skips that position's V slots.  Bytes are counted on the slot's barrier.
  constexpr int OKR = Sh::IRS * RB, OVR = (Sh::IRS + B) * RB;  // K, V row regions
  auto issue = [&](int s) {
    if (lane == 0) {
      const int4* dsc = ring.desc_at(s);
      if (dsc[0].x != -3) {
        uint8_t* st = ring.stage_at(s);
        uint64_t* bar = ring.bar_at(s);
        int4 qr[L::QR / 4];
        uint32_t qmask = 0;
#pragma unroll
        for (int q4 = 0; q4 < L::QR / 4; ++q4) {
          qr[q4] = ring.qset(s, q4);
          const bool any = qr[q4].x != p.N || qr[q4].y != p.N || qr[q4].z != p.N ||
                           qr[q4].w != p.N;
          qmask |= uint32_t(any) << q4;
        }
        fence_proxy_async();
        if constexpr (Sh::RES > 0) {
          constexpr int KS = (SE - 1) * G / 4;  // first 4-row set of the last edge position
          const int ne = qmask ? KS : B / 4;    // sets of edge rows in this stage
          // a starting stage: Q rows into the K slots of the last position,
          // zero-filled pad rows into its V slots (every V slot then holds a
          // real row or zeros, which the value sum below relies on)
          mbar_expect_tx(bar, (B / 4 + ne + __popc(qmask)) * L::SET_BYTES);
#pragma unroll
          for (int b4 = 0; b4 < B / 4; ++b4) {
            if (b4 < ne) {
              const int4 r = ring.eset(s, b4);
              L::gather(st + OKR, 4 * b4, &p.mk, r.x, r.y, r.z, r.w, bar);
              L::gather(st + OVR, 4 * b4, &p.mv, r.x, r.y, r.z, r.w, bar);
            } else {
              if ((qmask >> (b4 - KS)) & 1) {
                const int4 r = qr[b4 - KS];
                L::gather(st + OKR, 4 * b4, &p.mq, r.x, r.y, r.z, r.w, bar);
              }
              L::gather(st + OVR, 4 * b4, &p.mv, p.N, p.N, p.N, p.N, bar);
            }
          }
        } else {
          const uint32_t ibytes = L::IBULK ? item_rows<L>(qr[0], p.N) * RB
                                           : __popc(qmask) * L::SET_BYTES;
          mbar_expect_tx(bar, ibytes + 2 * (B / 4) * L::SET_BYTES);
          if constexpr (L::IBULK) {
            fetch_item_rows<L>(st, p.Q, qr[0], p.N, bar);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < L::QR / 4; ++q4)
              if ((qmask >> q4) & 1)
                L::gather(st, 4 * q4, &p.mq, qr[q4].x, qr[q4].y, qr[q4].z, qr[q4].w, bar);
          }
#pragma unroll
          for (int b4 = 0; b4 < B / 4; ++b4) {
            const int4 r = ring.eset(s, b4);
            L::gather(st + OKR, 4 * b4, &p.mk, r.x, r.y, r.z, r.w, bar);
            L::gather(st + OVR, 4 * b4, &p.mv, r.x, r.y, r.z, r.w, bar);
          }
        }
      }
    }
    __syncwarp();
    cp_async_commit();  // this iteration's index copies
  };

  // prologue: indices of stages 0..S-1, then rows of stages 0..S-2
  for (int s = 0; s < S; ++s) ring.generate(cur, s, lane);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int s = 0; s < S - 1; ++s) {
    ring.generate(cur, S + s, lane);
    issue(s);
  }

  float2 q[NC][PP], acc[NC][PP];
  float m[HL], l[HL];
  for (int i = 0;; ++i) {
    ring.generate(cur, i + 2 * S - 1, lane);
    __syncwarp();
    issue(i + S - 1);
    cp_async_wait<S - 1>();
    __syncwarp();
    const int4* dsc = ring.desc_at(i);
    if (dsc[0].x == -3) break;
    if (!__all_sync(FULL, ring.wait_rows(i, p.err, lane, ring.limit_at(i, p.fail_first_wait)))) break;
    const int4 d = dsc[g];
    const bool act = d.x >= 0;
    const int cnt = act ? (d.z & kCntMask) : 0;
    const uint8_t* st = ring.stage_at(i);

    if (act && (d.z & kFirst)) {
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int x = (t * NC + c) * 16;
        PR::load(lds16(Sh::RES ? st + OKR + L::off(Cur::slot(g, SE - 1), x) : st + L::offI(g, x)),
                 q[c]);
        if (!GAT) {
#pragma unroll
          for (int v = 0; v < PP; ++v) q[c][v] = f2mul(q[c][v], f2s(p.qmul));
        }
#pragma unroll
        for (int v = 0; v < PP; ++v) acc[c][v] = f2s(0.f);
      }
#pragma unroll
      for (int j = 0; j < HL; ++j) {
        m[j] = neg_inf();
        l[j] = 0.f;
      }
    }

    const uint8_t* ks = st + OKR;
    const uint8_t* vs = st + OVR;
    float sc[SE][HL];
#pragma unroll
    for (int k = 0; k < SE; ++k) {
      // slots past this group's count hold zero-filled pad rows or rows of an
      // earlier stage: their scores are discarded below, so they are read as is
      float2 a2[HL];
#pragma unroll
      for (int j = 0; j < HL; ++j) a2[j] = f2s(0.f);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 kr = lds16(ks + L::off(Cur::slot(g, k), (t * NC + c) * 16));
        float2 kf[PP];
        PR::load(kr, kf);
        float2& acc2 = a2[LH::of(c)];
        if (!GAT) {
#pragma unroll
          for (int v = 0; v < PP; ++v) acc2 = f2fma(q[c][v], kf[v], acc2);
        } else {
#pragma unroll
          for (int v = 0; v < PP; ++v) {
            const float2 z = f2add(q[c][v], kf[v]);
            acc2 = f2fma(ac1[c][v], z, f2fma(ac2[c][v], f2abs(z), acc2));
          }
        }
      }
      head_sums2<NC, CPH>(a2, sc[k]);
#pragma unroll
      for (int j = 0; j < HL; ++j) {
        if (GAT) sc[k][j] *= kLog2e;
        if (k >= cnt) sc[k][j] = neg_inf();
      }
    }
    if (act) {
      float corr[HL], base[HL];
#pragma unroll
      for (int j = 0; j < HL; ++j) {
        float mx = m[j];
#pragma unroll
        for (int k = 0; k < SE; ++k) mx = fmaxf(mx, sc[k][j]);  // -inf past the count
        base[j] = mx == neg_inf() ? 0.f : mx;
        corr[j] = ex2(m[j] - base[j]);
        l[j] *= corr[j];
        m[j] = mx;
      }
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int v = 0; v < PP; ++v) acc[c][v] = f2mul(acc[c][v], f2s(corr[LH::of(c)]));
      // branch-free for the dot score: past the count the score is -inf, so
      // the weight is 0, and the V slot holds a zero-filled pad row (or a
      // real row): the sum takes 0 there.  GATv2 keeps the branch.
#pragma unroll
      for (int k = 0; k < SE; ++k) {
        if (!GAT || k < cnt) {
          float pk[HL];
#pragma unroll
          for (int j = 0; j < HL; ++j) {
            pk[j] = ex2(sc[k][j] - base[j]);
            l[j] += pk[j];
          }
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            float2 vf[PP];
            PR::load(lds16(vs + L::off(Cur::slot(g, k), (t * NC + c) * 16)), vf);
#pragma unroll
            for (int v = 0; v < PP; ++v) acc[c][v] = f2fma(f2s(pk[LH::of(c)]), vf[v], acc[c][v]);
          }
        }
      }
    }

    // items that end in this stage; heavy chunks climb their node's merge tree
    const bool fin = act && (d.z & kLast);
    const bool heavy = fin && d.y < p.n_chunks;
    bool write = fin && !heavy;
    if (heavy) {
      auto store = [&](int slot) {
        float* pb = p.part + int64_t(slot) * p.pstride;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
#pragma unroll
          for (int v = 0; v < PP; v += 2)
            *reinterpret_cast<float4*>(pb + elem[c] + 2 * v) =
                make_float4(acc[c][v].x, acc[c][v].y, acc[c][v + 1].x, acc[c][v + 1].y);
        }
#pragma unroll
        for (int j = 0; j < HL; ++j)
          if (hw[j * LH::CPL]) {
            pb[HD + head[j * LH::CPL]] = m[j];
            pb[HD + p.H + head[j * LH::CPL]] = l[j];
          }
      };
      auto merge = [&](int c0, int cn) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int v = 0; v < PP; ++v) acc[c][v] = f2s(0.f);
#pragma unroll
        for (int j = 0; j < HL; ++j) {
          m[j] = neg_inf();
          l[j] = 0.f;
        }
        for (int kk = 0; kk < cn; kk += 4) {  // four children's loads in flight at a time
          float mo[4][HL], lo[4][HL];
          float4 f[4][NC][PP / 2];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const bool ok = kk + jj < cn;
            const float* pc = p.part + int64_t(c0 + (ok ? kk + jj : 0)) * p.pstride;
#pragma unroll
            for (int j = 0; j < HL; ++j) {
              mo[jj][j] = ok ? __ldcg(pc + HD + head[j * LH::CPL]) : neg_inf();
              lo[jj][j] = ok ? __ldcg(pc + HD + p.H + head[j * LH::CPL]) : 0.f;
            }
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
              for (int v = 0; v < PP / 2; ++v)
                f[jj][c][v] = ok ? __ldcg(reinterpret_cast<const float4*>(pc + elem[c] + 4 * v))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            float c1[HL], c2[HL];
#pragma unroll
            for (int j = 0; j < HL; ++j) {
              const float mn = fmaxf(m[j], mo[jj][j]);
              const float base = mn == neg_inf() ? 0.f : mn;
              c1[j] = ex2(m[j] - base);
              c2[j] = ex2(mo[jj][j] - base);
              l[j] = l[j] * c1[j] + lo[jj][j] * c2[j];
              m[j] = mn;
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              const float a1 = c1[LH::of(c)], a2 = c2[LH::of(c)];
#pragma unroll
              for (int v = 0; v < PP / 2; ++v) {
                acc[c][2 * v] = f2fma(acc[c][2 * v], f2s(a1),
                                      f2mul(make_float2(f[jj][c][v].x, f[jj][c][v].y), f2s(a2)));
                acc[c][2 * v + 1] = f2fma(acc[c][2 * v + 1], f2s(a1),
                                          f2mul(make_float2(f[jj][c][v].z, f[jj][c][v].w), f2s(a2)));
              }
            }
          }
        }
      };
      write = climb(p.tree, d.y, group_mask<TPR>(g), g * TPR, t == 0, merge, store);
    }
    if (write) {
      char* ob = static_cast<char*>(p.out) + int64_t(d.x) * RB;
      float inv[HL];
#pragma unroll
      for (int j = 0; j < HL; ++j) {
        inv[j] = l[j] > 0.f ? 1.f / l[j] : 0.f;
        if (hw[j * LH::CPL])
          p.lse[int64_t(d.x) * p.H + head[j * LH::CPL]] =
              l[j] > 0.f ? (m[j] + lg2(l[j])) * kLn2 : neg_inf();
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float2 o[PP];
#pragma unroll
        for (int v = 0; v < PP; ++v) o[v] = f2mul(acc[c][v], f2s(inv[LH::of(c)]));
        *reinterpret_cast<uint4*>(ob + (t * NC + c) * 16) = PR::store(o);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  ring.release(lane);
}

}  // namespace gattn
