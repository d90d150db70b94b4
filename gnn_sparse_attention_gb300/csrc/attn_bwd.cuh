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
  // row-gather maps (tma.cuh).  Pass 1: mi0..mi2 = Q, dO, O (item rows),
  // me0, me1 = K, V (edge rows), ms0 = lse (item stat rows).  Pass 2: mi0,
  // mi1 = K, V (item rows), me0, me1 = Q, dO (edge rows); the edges'
  // (lse log2(e), Delta) rows are copied by the lanes.
  CUtensorMap mi0, mi1, mi2, me0, me1, ms0;
  const int4* items;   // plan items (w = heavy id of a chunk)
  const int4* sorted;  // items by decreasing length
  int64_t n_items;
  int64_t n_chunks;    // items [0, n_chunks) are heavy chunks
  int N;               // rows; row index N is the zero-filled pad row
  const int32_t* idx;  // pass 1: CSR sources; pass 2: CSC destinations
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const void* dO;
  const float* lse;
  float* delta;        // [N, 2H] workspace: lse * log2(e) of the H heads, then Delta
  void* G1;            // pass 1: dQ;  pass 2: dK
  void* G2;            // pass 2: dV
  float* da;           // GATv2 [H*D] or null
  const float* a;
  float qmul;          // DOT: scale * log2(e)
  float scale;         // DOT: scale
  float slope;
  int H, D;
  int rows16;          // lse rows are gathered by TMA (H % 4 == 0, lse 16-B aligned)
  float* part;         // partials per tree slot: pass 1 [slots][HD], pass 2 [slots][2*HD]
  Tree tree;           // merge trees of the heavy items of this pass
  float* da_part;      // [gridDim.x][HD]
  int32_t* da_cnt;
  int32_t* err;        // set when a wait gives up
  int fail_first_wait; // nonzero: every warp's first wait expires at once (failure-path test)
};

// Largest per-node fp32 row (lse or Delta): H <= RB/16 floats, padded to 16 B.
template <int RB>
struct StatBytes {
  static constexpr int value = RB / 4 < 16 ? 16 : RB / 4;
};

template <typename T, int RB, int SB>
struct CsrShape {
  using L = Lay<T, RB, SB>;
  static constexpr int LS = StatBytes<RB>::value;
  // Item rows inline (attn_pipe.cuh, BundleCursor) where a stage holds whole
  // 4-row sets and at least 4 edges per item: a starting item's Q and dO
  // rows take its group's K and V slots of the last edge position, its O row
  // the K slot of the one before.  Otherwise the Q, dO and O rows have a
  // region of their own (IR slots each).
  static constexpr int RES = (L::G >= 4 && L::SE >= 4) ? 2 : 0;
  static constexpr int IRS = RES ? 0 : L::IR;
  // [IRS Q, dO, O rows] [lse sets] [B K rows] [B V rows]
  static constexpr int OL = 3 * IRS * RB;               // lse sets
  static constexpr int OK = OL + L::QR / 4 * L::SSB;    // K rows
  static constexpr int OV = OK + L::B * RB;             // V rows
  static constexpr int STAGE = OV + L::B * RB;
  static constexpr int WARP_BYTES = align128(kStages * STAGE + L::META);
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int MINB = WarpsFor<WARP_BYTES>::minb;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

template <typename T, int RB, int SB, int DB>
struct CscShape {
  using L = Lay<T, RB, SB>;
  static constexpr int H = RB / DB;                     // heads
  // Item rows inline where a stage holds whole 4-row sets and at least 4
  // edges per item: a starting item's K and V rows take its group's Q and dO
  // slots of the last edge position.  Otherwise K and V rows have a region
  // of their own.
  static constexpr int RES = (L::G >= 4 && L::SE >= 4) ? 1 : 0;
  static constexpr int IRS = RES ? 0 : L::IR;
  // [IRS K, V rows] [B Q rows] [B dO rows] [B (lse log2 e, Delta) rows]
  static constexpr int SROW = 8 * H;                    // bytes of one (lse, Delta) row
  static constexpr int OQE = 2 * IRS * RB;              // Q rows of the edges
  static constexpr int OGE = OQE + L::B * RB;           // dO rows
  static constexpr int OLS = OGE + L::B * RB;           // (lse, Delta) rows
  static constexpr int STAGE = align128(OLS + L::B * SROW);
  static constexpr int WARP_BYTES = align128(kStages * STAGE + L::META);
  static constexpr int WARPS = WarpsFor<WARP_BYTES>::value;
  static constexpr int MINB = WarpsFor<WARP_BYTES>::minb;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SMEM = WARPS * WARP_BYTES;
};

// Copy the fp32 rows src + node_r * H (r < n, node_r < 0: skip) into the
// stat-set layout (row r at set r / 4, slot r % 4, H floats a row) with 4-byte cp.async, node_r taken from lane r of
// `nodes` (the fallback when the rows are not whole 16-byte pieces).
// Uniform trip count.
template <int SSB>
__device__ __forceinline__ void copy_stat_rows(uint8_t* dst, const float* src, int nodes, int n,
                                               int H, int lane) {
  constexpr unsigned FULL = 0xffffffffu;
  const int trips = (n * H + 31) / 32;
  for (int tr = 0; tr < trips; ++tr) {
    const int x = tr * 32 + lane;
    const int r = x / H, f = x % H;
    const int i = __shfl_sync(FULL, nodes, r & 31);
    if (x < n * H && i >= 0)
      cp_async4(dst + (r / 4) * SSB + ((r % 4) * H + f) * 4, src + int64_t(i) * H + f);
  }
}

// ---------------------------------------------------------------------------
// pass 1: CSR
// ---------------------------------------------------------------------------
template <typename T, int RB, int DB, int KIND, int SB>
__global__ void __launch_bounds__(CsrShape<T, RB, SB>::THREADS, min_blocks<CsrShape<T, RB, SB>::WARP_BYTES, RB, SB>(KIND)) bwd_csr_kernel(const __grid_constant__ BwdParams p) {
  using L = Lay<T, RB, SB>;
  using Sh = CsrShape<T, RB, SB>;
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
  using Cur = BundleCursor<G, SE, Sh::RES>;
  Cur cur;
  cur.start(p.sorted, p.n_items, p.idx, p.N, warp, nwarps, ring.items, lane);

  // stage: [IRS][Q row] [IRS][dO row] [IRS][O row] [QR/4][lse set] [B][K row]
  // [B][V row].  TMA gathers from lane 0 (item rows only for 4-row sets that
  // hold a starting item, pad row N elsewhere; with fewer than 4 groups a
  // warp copies just the starting items' rows; inline item rows go to the
  // K / V slots of the last two edge positions of a stage that starts a
  // bundle); lse rows by gather when they are whole 16-byte pieces, else by
  // 4-byte cp.async.
  constexpr int OQ = 0, ODO = Sh::IRS * RB, OO = 2 * Sh::IRS * RB;
  constexpr int OL = Sh::OL, OK = Sh::OK, OV = Sh::OV;
  // inline: slots of a starting item's Q / dO rows (last edge position) and O row
  constexpr int K1 = (SE - 1) * G / 4, K2 = (SE - 2) * G / 4;
  auto issue = [&](int s) {
    const int4* dsc = ring.desc_at(s);
    if (lane == 0 && dsc[0].x != -3) {
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
      const uint32_t ibytes = L::IBULK ? item_rows<L>(qr[0], p.N) * 3 * RB
                                       : __popc(qmask) * 3 * L::SET_BYTES;
      // inline: a stage that starts a bundle gathers edge rows only below K2
      const int ne = (Sh::RES > 0 && qmask) ? K2 : B / 4;
      fence_proxy_async();
      mbar_expect_tx(bar, ibytes + (p.rows16 ? __popc(qmask) * 16 * p.H : 0) +
                              2 * ne * L::SET_BYTES);
#pragma unroll
      for (int q4 = 0; q4 < L::QR / 4; ++q4)
        if ((qmask >> q4) & 1) {
          const int4 r = qr[q4];
          if constexpr (Sh::RES > 0) {
            L::gather(st + OK, 4 * (K1 + q4), &p.mi0, r.x, r.y, r.z, r.w, bar);
            L::gather(st + OV, 4 * (K1 + q4), &p.mi1, r.x, r.y, r.z, r.w, bar);
            L::gather(st + OK, 4 * (K2 + q4), &p.mi2, r.x, r.y, r.z, r.w, bar);
          } else if constexpr (L::IBULK) {
            fetch_item_rows<L>(st + OQ, p.Q, r, p.N, bar);
            fetch_item_rows<L>(st + ODO, p.dO, r, p.N, bar);
            fetch_item_rows<L>(st + OO, p.O, r, p.N, bar);
          } else {
            L::gather(st + OQ, 4 * q4, &p.mi0, r.x, r.y, r.z, r.w, bar);
            L::gather(st + ODO, 4 * q4, &p.mi1, r.x, r.y, r.z, r.w, bar);
            L::gather(st + OO, 4 * q4, &p.mi2, r.x, r.y, r.z, r.w, bar);
          }
          if (p.rows16) tma_gather4(st + OL + q4 * L::SSB, &p.ms0, 0, r.x, r.y, r.z, r.w, bar);
        }
#pragma unroll
      for (int b4 = 0; b4 < B / 4; ++b4) {
        if (b4 < ne) {
          const int4 r = ring.eset(s, b4);
          L::gather(st + OK, 4 * b4, &p.me0, r.x, r.y, r.z, r.w, bar);
          L::gather(st + OV, 4 * b4, &p.me1, r.x, r.y, r.z, r.w, bar);
        }
      }
    }
    if (!p.rows16) {  // lse rows of starting items by 4-byte copies
      const int4 dg = lane < G ? dsc[lane] : make_int4(-1, 0, 0, 0);
      const int fnode = (dsc[0].x != -3 && lane < G && dg.x >= 0 && (dg.z & kFirst)) ? dg.x : -1;
      copy_stat_rows<L::SSB>(ring.stage_at(s) + OL, p.lse, fnode, G, p.H, lane);
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

  float2 q[NC][PP], gq[NC][PP], dq[NC][PP];
  float lse2[HL], dlt[HL];
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
    const bool first = act && (d.z & kFirst);

    if (__any_sync(FULL, first)) {
      // item start: q, dO, Delta = dO . O, lse (every lane joins the head
      // reduction).  Delta is summed in exactly the order of every dp = dO . v
      // below and in the CSC pass, so that dp - Delta is exactly 0 wherever
      // out equals a single neighbour's v (a one-edge row).
      float dsum[HL];
      float2 a2[HL];
#pragma unroll
      for (int j = 0; j < HL; ++j) a2[j] = f2s(0.f);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float2 o[PP];
        if (first) {
          const int x = (t * NC + c) * 16;
          if constexpr (Sh::RES > 0) {
            const int xa = L::off(Cur::slot(g, SE - 1), x), xb = L::off(Cur::slot(g, SE - 2), x);
            PR::load(lds16(st + OK + xa), q[c]);
            PR::load(lds16(st + OV + xa), gq[c]);
            PR::load(lds16(st + OK + xb), o);
          } else {
            const int xi = L::offI(g, x);
            PR::load(lds16(st + OQ + xi), q[c]);
            PR::load(lds16(st + ODO + xi), gq[c]);
            PR::load(lds16(st + OO + xi), o);
          }
        } else {
#pragma unroll
          for (int v = 0; v < PP; ++v) o[v] = f2s(0.f);
        }
#pragma unroll
        for (int v = 0; v < PP; ++v)
          a2[LH::of(c)] = f2fma(first ? gq[c][v] : f2s(0.f), o[v], a2[LH::of(c)]);
      }
      head_sums2<NC, CPH>(a2, dsum);
      if (first) {
        const float* ls = reinterpret_cast<const float*>(st + OL + (g / 4) * L::SSB) + (g % 4) * p.H;
#pragma unroll
        for (int j = 0; j < HL; ++j) {
          const int c0 = j * LH::CPL;
          dlt[j] = dsum[j];
          lse2[j] = ls[head[c0]] * kLog2e;
          // the CSC pass reads (lse log2(e), Delta) of a destination as one
          // row; every chunk of a heavy node computes the same values:
          // duplicate writes store identical values
          if (hw[c0]) {
            float* srow = p.delta + int64_t(d.x) * 2 * p.H;
            srow[head[c0]] = lse2[j];
            srow[p.H + head[c0]] = dlt[j];
          }
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          if (!GAT) {
#pragma unroll
            for (int v = 0; v < PP; ++v) q[c][v] = f2mul(q[c][v], f2s(p.qmul));
          }
#pragma unroll
          for (int v = 0; v < PP; ++v) dq[c][v] = f2s(0.f);
        }
      }
    }

    const uint8_t* ks = st + OK;
    const uint8_t* vs = st + OV;
#pragma unroll
    for (int k = 0; k < SE; ++k) {
      const bool valid = k < cnt;
      // slots past this group's count are read as they are (zero-filled pad
      // rows or rows of an earlier stage): nothing below uses their results
      float sc[HL], dp[HL];
      float2 s2[HL], p2[HL];
#pragma unroll
      for (int j = 0; j < HL; ++j) s2[j] = p2[j] = f2s(0.f);
      float2 kf[NC][PP];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int off = L::off(Cur::slot(g, k), (t * NC + c) * 16);
        float2 vf[PP];
        PR::load(lds16(ks + off), kf[c]);
        PR::load(lds16(vs + off), vf);
        const int j = LH::of(c);
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          p2[j] = f2fma(gq[c][v], vf[v], p2[j]);
          if (!GAT) {
            s2[j] = f2fma(q[c][v], kf[c][v], s2[j]);
          } else {
            const float2 z = make_float2(q[c][v].x + kf[c][v].x, q[c][v].y + kf[c][v].y);
            const float2 lr = make_float2(z.x > 0.f ? z.x : p.slope * z.x,
                                          z.y > 0.f ? z.y : p.slope * z.y);
            s2[j] = f2fma(av[c][v], lr, s2[j]);
          }
        }
      }
      head_sums2<NC, CPH>(s2, sc);
      head_sums2<NC, CPH>(p2, dp);
      // dot score branch-free: ds is 0 for a slot past the group's count (a
      // select, so whatever such a slot's rows hold never reaches the sums);
      // GATv2 keeps the branch (its longer body spills without it)
      if (!GAT || (act && valid)) {
        const bool use = act && valid;
        float ds[HL];
#pragma unroll
        for (int j = 0; j < HL; ++j) {
          const float pr = ex2((GAT ? sc[j] * kLog2e : sc[j]) - lse2[j]);
          ds[j] = use ? pr * (dp[j] - dlt[j]) : 0.f;
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float dsc_ = ds[LH::of(c)];
          if (!GAT) {
#pragma unroll
            for (int v = 0; v < PP; ++v) dq[c][v] = f2fma(f2s(dsc_), kf[c][v], dq[c][v]);
          } else {
#pragma unroll
            for (int v = 0; v < PP; ++v) {
              const float2 z = make_float2(q[c][v].x + kf[c][v].x, q[c][v].y + kf[c][v].y);
              const float2 sg = make_float2(z.x > 0.f ? 1.f : p.slope, z.y > 0.f ? 1.f : p.slope);
              const float2 lr = make_float2(z.x > 0.f ? z.x : p.slope * z.x,
                                            z.y > 0.f ? z.y : p.slope * z.y);
              dq[c][v] = f2fma(f2mul(f2s(dsc_), av[c][v]), sg, dq[c][v]);
              dacc[c][v] = f2fma(f2s(dsc_), lr, dacc[c][v]);
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
    int& s_last = *reinterpret_cast<int*>(smem + Sh::WARPS * HD * 4);
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
template <typename T, int RB, int DB, int KIND, int SB>
__global__ void __launch_bounds__(CscShape<T, RB, SB, DB>::THREADS, min_blocks<CscShape<T, RB, SB, DB>::WARP_BYTES, RB, SB>(KIND)) bwd_csc_kernel(const __grid_constant__ BwdParams p) {
  using L = Lay<T, RB, SB>;
  using Sh = CscShape<T, RB, SB, DB>;
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
  const float gc1 = 0.5f * (1.f + p.slope), gc2 = 0.5f * (1.f - p.slope);  // LReLU = c1 z + c2 |z|

  const int64_t warp = (int64_t(blockIdx.x) * Sh::THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * Sh::THREADS) >> 5;
  using Cur = BundleCursor<G, SE, Sh::RES>;
  Cur cur;
  cur.start(p.sorted, p.n_items, p.idx, p.N, warp, nwarps, ring.items, lane);

  // stage: [IRS][K row] [IRS][V row] [B][Q row] [B][dO row] [B][(lse log2 e,
  // Delta) row].  TMA gathers from lane 0 (pad row N in unused slots; with
  // fewer than 4 groups a warp copies just the starting items' rows; inline
  // item rows go to the Q / dO slots of the last edge position of a stage
  // that starts a bundle).  The 8H-byte statistic rows of the edges are
  // copied by the lanes with cp.async (16-byte pieces; 8 bytes when H = 1):
  // many small independent copies are cheaper there than row gathers.
  constexpr int OKI = 0, OVI = Sh::IRS * RB;
  constexpr int OQE = Sh::OQE, OGE = Sh::OGE, OLS = Sh::OLS;
  constexpr int SROW = Sh::SROW;
  constexpr int PB = SROW < 16 ? SROW : 16;   // bytes of one statistic piece
  constexpr int PPR = SROW / PB;             // pieces per row
  constexpr int K1 = (SE - 1) * G / 4;       // inline: first set of the last edge position
  auto issue = [&](int s) {
    const int4* dsc = ring.desc_at(s);
    const bool live = dsc[0].x != -3;
    if (lane == 0 && live) {
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
      const uint32_t ibytes = L::IBULK ? item_rows<L>(qr[0], p.N) * 2 * RB
                                       : __popc(qmask) * 2 * L::SET_BYTES;
      const int ne = (Sh::RES > 0 && qmask) ? K1 : B / 4;  // sets of edge rows
      fence_proxy_async();
      mbar_expect_tx(bar, ibytes + 2 * ne * L::SET_BYTES);
#pragma unroll
      for (int q4 = 0; q4 < L::QR / 4; ++q4)
        if ((qmask >> q4) & 1) {
          const int4 r = qr[q4];
          if constexpr (Sh::RES > 0) {
            L::gather(st + OQE, 4 * (K1 + q4), &p.mi0, r.x, r.y, r.z, r.w, bar);
            L::gather(st + OGE, 4 * (K1 + q4), &p.mi1, r.x, r.y, r.z, r.w, bar);
          } else if constexpr (L::IBULK) {
            fetch_item_rows<L>(st + OKI, p.K, r, p.N, bar);
            fetch_item_rows<L>(st + OVI, p.V, r, p.N, bar);
          } else {
            L::gather(st + OKI, 4 * q4, &p.mi0, r.x, r.y, r.z, r.w, bar);
            L::gather(st + OVI, 4 * q4, &p.mi1, r.x, r.y, r.z, r.w, bar);
          }
        }
#pragma unroll
      for (int b4 = 0; b4 < B / 4; ++b4) {
        if (b4 < ne) {
          const int4 r = ring.eset(s, b4);
          L::gather(st + OQE, 4 * b4, &p.me0, r.x, r.y, r.z, r.w, bar);
          L::gather(st + OGE, 4 * b4, &p.me1, r.x, r.y, r.z, r.w, bar);
        }
      }
    }
    if (live) {  // statistic rows of the stage's edges (pad slots skipped)
      uint8_t* sd = ring.stage_at(s) + OLS;
      const int* ixs = ring.ix_at(s);
      for (int x = lane; x < B * PPR; x += 32) {
        const int b = x / PPR, pc = x % PPR;
        const int j = ixs[b];
        if (j != p.N) {
          const float* src = p.delta + int64_t(j) * 2 * Sh::H + pc * (PB / 4);
          if constexpr (PB == 16) cp_async16(sd + b * SROW + pc * PB, src);
          else cp_async8(sd + b * SROW + pc * PB, src);
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

  // dk: the dot score's dK sum; GATv2: sum of ds over z > 0 per element,
  // with s1 the per-head sum of ds (combined at the item's end)
  float2 k[NC][PP], vv[NC][PP], dk[NC][PP], dv[NC][PP];
  float s1[GAT ? HL : 1];
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
        if constexpr (Sh::RES > 0) {
          const int xa = L::off(Cur::slot(g, SE - 1), x);
          PR::load(lds16(st + OQE + xa), k[c]);
          PR::load(lds16(st + OGE + xa), vv[c]);
        } else {
          PR::load(lds16(st + OKI + L::offI(g, x)), k[c]);
          PR::load(lds16(st + OVI + L::offI(g, x)), vv[c]);
        }
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          if (!GAT) k[c][v] = f2mul(k[c][v], f2s(p.qmul));
          dk[c][v] = dv[c][v] = f2s(0.f);
        }
      }
      if (GAT) {
#pragma unroll
        for (int j = 0; j < HL; ++j) s1[j] = 0.f;
      }
    }

    const uint8_t* qs = st + OQE;
    const uint8_t* gs = st + OGE;

#pragma unroll
    for (int e = 0; e < SE; ++e) {
      const bool valid = e < cnt;
      // slots past this group's count are read as they are (zero-filled pad
      // rows or rows of an earlier stage): nothing below uses their results
      float sc[HL], dp[HL];
      float2 s2[HL], p2[HL];
#pragma unroll
      for (int j = 0; j < HL; ++j) s2[j] = p2[j] = f2s(0.f);
      float2 qf[NC][PP], gf[NC][PP];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int off = L::off(Cur::slot(g, e), (t * NC + c) * 16);
        PR::load(lds16(qs + off), qf[c]);
        PR::load(lds16(gs + off), gf[c]);
        const int j = LH::of(c);
#pragma unroll
        for (int v = 0; v < PP; ++v) {
          p2[j] = f2fma(gf[c][v], vv[c][v], p2[j]);
          if (!GAT) {
            s2[j] = f2fma(qf[c][v], k[c][v], s2[j]);
          } else {  // qf becomes z = xl_i + xr_j
            qf[c][v] = f2add(qf[c][v], k[c][v]);
            const float2 lr = f2fma(f2s(gc1), qf[c][v], f2mul(f2s(gc2), f2abs(qf[c][v])));
            s2[j] = f2fma(av[c][v], lr, s2[j]);
          }
        }
      }
      head_sums2<NC, CPH>(s2, sc);
      head_sums2<NC, CPH>(p2, dp);
      // dot score branch-free: p and ds are 0 for a slot past the group's
      // count (a select, so whatever such a slot's rows hold never reaches
      // the sums); GATv2 keeps the branch
      if (!GAT || (act && valid)) {
        const bool use = act && valid;
        const float* srow = reinterpret_cast<const float*>(st + OLS + Cur::slot(g, e) * SROW);
        float pr[HL], ds[HL];
#pragma unroll
        for (int j = 0; j < HL; ++j) {
          const int hh = head[j * LH::CPL];
          const float ls2 = srow[hh];
          const float dl = srow[Sh::H + hh];
          const float pe = ex2((GAT ? sc[j] * kLog2e : sc[j]) - ls2);
          pr[j] = use ? pe : 0.f;
          ds[j] = use ? pe * (dp[j] - dl) : 0.f;
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float prc = pr[LH::of(c)], dsc_ = ds[LH::of(c)];
#pragma unroll
          for (int v = 0; v < PP; ++v) dv[c][v] = f2fma(f2s(prc), gf[c][v], dv[c][v]);
          if (!GAT) {
#pragma unroll
            for (int v = 0; v < PP; ++v) dk[c][v] = f2fma(f2s(dsc_), qf[c][v], dk[c][v]);
          } else {
#pragma unroll
            for (int v = 0; v < PP; ++v) {
              const float2 z = qf[c][v];
              dk[c][v] = f2add(dk[c][v], make_float2(z.x > 0.f ? dsc_ : 0.f, z.y > 0.f ? dsc_ : 0.f));
            }
          }
        }
        if (GAT) {
#pragma unroll
          for (int j = 0; j < HL; ++j) s1[j] += ds[j];
        }
      }
    }

    const bool fin = act && (d.z & kLast);
    if (GAT && fin) {  // dXr = a (s sum ds + (1 - s) sum_{z > 0} ds)
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int v = 0; v < PP; ++v)
          dk[c][v] = f2mul(av[c][v], f2fma(f2s(1.f - p.slope), dk[c][v],
                                           f2s(p.slope * s1[LH::of(c)])));
    }
    const bool heavy = fin && d.y < p.n_chunks;
    bool write = fin && !heavy;
    if (heavy) {
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
