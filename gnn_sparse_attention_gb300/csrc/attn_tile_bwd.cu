// attn_tile_bwd.cu -- dense-tile backward on the tensor cores (tcgen05 + TMEM).
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", attention-based layers: the backward
// pass recomputes the attention weights from the cached log-sum-exp, and
// locally dense neighbourhoods packed into block tiles become dense matrix
// products on the tensor cores.
//
// For the edges of a tile (row block I, column block J, bit mask), with
// p_ij = exp(s_ij - lse_i) and ds_ij = p_ij (dO_i . v_j - Delta_i):
//   row kernel    (one row block at a time):    dQ_I += scale * dS K_J
//   column kernel (one column block at a time): dV_J += P^T dO_I
//                                               dK_J += scale * dS^T Q_I
// Both recompute their 128 x 128 block of scores and of dO . v on the
// tensor cores -- the row kernel S = Q K^T and dP = dO V^T, the column
// kernel the transposes S^T = K Q^T and dP^T = V dO^T, so that TMEM lane r
// is always row r of the own block.  16 warps split each lane's 128 columns
// into four 32-column chunks (a warp reads only its own lane quarter); a
// thread forms p and ds in fp32 from the forward's lse and the
// destination's Delta (written by the residual CSR pass) and stores them as
// bf16 operand tiles in shared memory (the 128-byte swizzled K-major layout
// the TMA loads use); one thread issues the gradient products.  The
// residual passes (CSR for dQ, CSC for dK and dV, over the edges outside
// the tiles) run first and write every row; after a block's last tile of a
// head, the tile kernels add their part in fp32 to those rows -- brought in
// as TMA tiles into the step's own-block operand region, which the score
// products no longer need -- and store the bf16 sums back with TMA.
//
// Schedule: one CTA per SM walks its blocks (grid stride), the heads, and
// the block's tiles, steered by the plan's per-tile step descriptors
// (loaded two steps ahead).  With two operand slots (D = 64) the next
// step's TMA loads (four 128 x D operand tiles and the 2 KB mask) are in
// flight while the current step computes.  TMEM holds S [0, 128), dP
// [128, 256) and the gradient accumulators from column 256 (row kernel dQ;
// column kernel dV, then dK), which sum over the tiles of a block and head.
// Every mbarrier wait is bounded; a wait that gives up sets the plan's error
// word, the block drains what it issued (again bounded), frees its TMEM and
// returns.
#include <cuda.h>

#include "attn_pipe.cuh"
#include "attn_tile.cuh"
#include "tcgen05.cuh"

namespace gattn {

namespace {

constexpr int kT = kTileRows;        // rows / columns of a tile
constexpr int kWarps = 16;           // four warps per TMEM lane quarter
constexpr int kThr = kWarps * 32;    // thread (row r, chunk c): row r of the own block,
                                     // columns [32c, 32c + 32) of the 128-wide blocks
constexpr int kTB = kT * 128;        // one 128 x 64 bf16 operand tile (16 KB)
constexpr int kMaskB = kT * 16;      // 128 rows x 4 mask words
constexpr uint32_t kCols = 512;      // TMEM columns

// Shared memory of one CTA: NS operand slots [A0 A1 B0 B1 mask], the
// thread-written operand tiles, the other block's statistics (column
// kernel) and the barriers.
template <int D, int NS, bool COL>
struct BwdSmem {
  static constexpr int KB = D / 64;                     // 64-column pieces of a head
  static constexpr int A0 = 0;                          // own block:   Q (row) / K (column)
  static constexpr int A1 = KB * kTB;                   // own block:   dO (row) / V (column)
  static constexpr int B0 = 2 * KB * kTB;               // other block: K (row) / Q (column)
  static constexpr int B1 = 3 * KB * kTB;               // other block: V (row) / dO (column)
  static constexpr int MASK = 4 * KB * kTB;
  static constexpr int SLOT = MASK + kMaskB;
  static constexpr int W0 = NS * SLOT;                  // dS (row) / P^T (column)
  static constexpr int W1 = W0 + 2 * kTB;               // dS^T (column)
  static constexpr int STAT = W1 + (COL ? 2 * kTB : 0); // lse * log2(e), Delta of the other block
  static constexpr int BAR = STAT + (COL ? 2 * kT * 4 : 0);
  static constexpr int END = BAR + 64;
  static constexpr int BYTES = END + 1024;              // slack to align the base to 1024
  static_assert(SLOT % 1024 == 0 && W0 % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
  static_assert(BYTES <= 227 * 1024, "shared memory of one CTA");
};

// out = acc * mul + residual (8 bf16 values)
__device__ __forceinline__ uint4 add_rounded(const float* acc, float mul, uint4 res) {
  const uint32_t in[4] = {res.x, res.y, res.z, res.w};
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float r0 = __uint_as_float(in[q] << 16), r1 = __uint_as_float(in[q] & 0xffff0000u);
    w[q] = tc::bf16x2_bits(fmaf(acc[2 * q], mul, r0), fmaf(acc[2 * q + 1], mul, r1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

template <int D, int NS, bool COL>
__global__ void __launch_bounds__(kThr, 1) tile_bwd_kernel(const __grid_constant__ TileBwdParams p) {
  using namespace tc;
  using SM = BwdSmem<D, NS, COL>;
  constexpr int KB = SM::KB;
  constexpr uint32_t IDESC_S = f16_idesc(kT, kT, false);
  constexpr uint32_t IDESC_G = f16_idesc(kT, 64, true);  // one 64-column piece of a gradient
  constexpr uint32_t LOAD_BYTES = 4 * KB * kTB + kMaskB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* barL = reinterpret_cast<uint64_t*>(smem + SM::BAR);  // [2] operand slots
  uint64_t* barS = barL + 2;
  uint64_t* barD = barL + 3;
  uint64_t* barR = barL + 4;  // residual tiles of the epilogue
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(barL + 5);
  float* sL = reinterpret_cast<float*>(smem + SM::STAT);  // column kernel only
  float* sDl = sL + kT;

  const int tid = threadIdx.x, warp = tid >> 5;
  // warp w reads TMEM lanes [32 (w % 4), + 32) (a warp may only touch its
  // lane quarter) and owns the 32-column chunk cc = w / 4 of those rows
  const int r = (warp & 3) * 32 + (tid & 31);
  const int cc = warp >> 2;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(barL + s, 1);
    mbar_init(barS, 1);
    mbar_init(barD, 1);
    mbar_init(barR, 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
            smem_u32(sTmem)),
        "r"(kCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem, tP = tmem + kT, tG = tmem + 2 * kT, tG2 = tmem + 2 * kT + D;
  const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter

  // TMA loads of one step (descriptor d) into slot s (thread 0)
  auto issue = [&](const TileStep& c, int4 d, int s) {
    uint8_t* sl = smem + s * SM::SLOT;
    fence_proxy_async();
    mbar_expect_tx(barL + s, LOAD_BYTES);
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const int x = c.h * D + kb * 64;
      tma_tile2d(sl + SM::A0 + kb * kTB, &p.ma0, x, d.x * kT, barL + s);
      tma_tile2d(sl + SM::A1 + kb * kTB, &p.ma1, x, d.x * kT, barL + s);
      tma_tile2d(sl + SM::B0 + kb * kTB, &p.mb0, x, d.y * kT, barL + s);
      tma_tile2d(sl + SM::B1 + kb * kTB, &p.mb1, x, d.y * kT, barL + s);
    }
    bulk_g2s(sl + SM::MASK, p.mask + int64_t(d.z) * kT * 4, kMaskB, barL + s);
  };

  // barrier phases: bit s of phL = parity of slot s's next completion;
  // bit s of pendL = a load into slot s is in flight
  uint32_t phL = 0, pendL = 0, nS = 0, nD = 0, nR = 0;
  bool pendS = false, pendD = false, pendR = false;
  bool bad = false;

  // lse * log2(e) and Delta of row r of the rows a step's scores belong to
  // (row kernel: the own block; column kernel: the tile's row block)
  auto stats = [&](const TileStep& c, int4 d, float& a, float& b) {
    const int i = (COL ? d.y : d.x) * kT + r;
    a = 0.f;
    b = 0.f;
    if (i < p.N) {
      a = p.lse[int64_t(i) * p.H + c.h] * kLog2e;
      b = p.delta[int64_t(i) * 2 * p.H + p.H + c.h];
    }
  };
  // The epilogue's 32-column pieces: NG gradient tensors (row kernel dQ;
  // column kernel dV, dK) of D / 32 pieces each; thread chunk cc takes
  // pieces cc, cc + 4, ...  Piece x is tensor t = x / (D / 32), columns
  // 32 (x % (D / 32)) of the head row.  Tensor t's residual tile (rows the
  // CSR / CSC pass wrote) arrives by TMA in the slot's own-block operand
  // region, free once S and dP are done (t = 0 in A0, t = 1 in A1, swizzled
  // like every operand tile); the sums are written back in place and leave
  // by TMA stores, so no thread touches global memory in the epilogue.
  constexpr int NG = COL ? 2 : 1;
  constexpr int NPC = NG * D / 32;
  constexpr int NPT = (NPC + 3) / 4;  // pieces per thread (at most)
  auto gmap = [&](int t) -> const CUtensorMap* { return (COL && t == 0) ? &p.mg2 : &p.mg1; };
  auto load_res = [&](uint8_t* sl, int own, int h) {  // thread 0
    fence_proxy_async();
    mbar_expect_tx(barR, NG * KB * kTB);
#pragma unroll
    for (int t = 0; t < NG; ++t)
#pragma unroll
      for (int kb = 0; kb < KB; ++kb)
        tma_tile2d(sl + (t ? SM::A1 : SM::A0) + kb * kTB, gmap(t), h * D + kb * 64, own * kT, barR);
  };
  auto epilogue = [&](uint8_t* sl) {
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int x = cc + 4 * j;
      if (x < NPC) {  // warp-uniform: the TMEM load is a whole-warp instruction
        const int t = x / (D / 32), col = (x % (D / 32)) * 32;
        float a[32];
        tmem_ld32((t ? tG2 : tG) + lane_off + col, a);
        tmem_wait_ld();
        uint8_t* row = sl + (t ? SM::A1 : SM::A0) + (col / 64) * kTB + r * 128;
        const float mul = (COL && t == 0) ? 1.f : p.scale;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4* ptr = reinterpret_cast<uint4*>(row + ((((col % 64) / 8 + q) ^ (r & 7)) * 16));
          *ptr = add_rounded(a + 8 * q, mul, *ptr);
        }
      }
    }
  };
  auto store_res = [&](const uint8_t* sl, int own, int h) {  // thread 0
#pragma unroll
    for (int t = 0; t < NG; ++t)
#pragma unroll
      for (int kb = 0; kb < KB; ++kb)
        tma_store2d(gmap(t), h * D + kb * 64, own * kT, sl + (t ? SM::A1 : SM::A0) + kb * kTB);
    bulk_commit();
  };

  // Step k: wait for its operands -> S, dP products (then the residual
  // tiles' loads when the step ends a (block, head)) -> p, ds -> the
  // gradient products -> the epilogue.  Descriptors are loaded two steps
  // ahead and statistics one step ahead, so no dependent chain of small
  // loads sits on a step's critical path.
  TileStep cur{-1, 0, 0, 0, -1}, nx{-1, 0, 0, 0, -1};
  int4 dc = make_int4(0, 0, 0, 0), dn = make_int4(0, 0, 0, 0);
  if (blockIdx.x < p.n_grp) {
    cur = tile_step_block(p, blockIdx.x, p.grp_ptr[blockIdx.x]);
    dc = p.desc[cur.q];
    nx = tile_step_after(p, cur, dc);
    if (nx.g >= 0) dn = p.desc[nx.q];
  }
  float nl = 0.f, nd = 0.f;      // statistics of `cur`, fetched a step ahead
  if (cur.g >= 0) {
    if (tid == 0) issue(cur, dc, 0);
    pendL = 1u;
    stats(cur, dc, nl, nd);
  }
  for (int k = 0; cur.g >= 0; ++k) {
    const int s = NS == 2 ? (k & 1) : 0;
    const bool more = nx.g >= 0;
    const TileStep n2 = more ? tile_step_after(p, nx, dn) : TileStep{-1, 0, 0, 0, -1};
    const int4 d2 = n2.g >= 0 ? p.desc[n2.q] : make_int4(0, 0, 0, 0);  // used next step
    const bool first = dc.w & 1;
    const bool last = dc.w & 2;
    if constexpr (NS == 2) {
      if (more) {
        // slot s ^ 1 was released by the previous step once its epilogue's
        // stores have read their tiles
        if (tid == 0) {
          bulk_wait_read();
          issue(nx, dn, s ^ 1);
        }
        pendL |= 1u << (s ^ 1);
      }
    }
    const float lse2 = nl, dl = nd;
    if constexpr (COL) {  // the previous step's reads of sL / sDl ended before its mid-step barrier
      if (cc == 0) {
        sL[r] = lse2;
        sDl[r] = dl;
      }
    }
    if (more) stats(nx, dn, nl, nd);
    bool ok = mbar_wait(barL + s, (phL >> s) & 1u);
    if (__syncthreads_or(!ok)) { bad = true; break; }
    phL ^= 1u << s;
    pendL &= ~(1u << s);

    // ---- S and dP (row kernel: Q K^T, dO V^T; column kernel: K Q^T, V dO^T)
    uint8_t* sl = smem + s * SM::SLOT;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k2 = 0; k2 < D / 16; ++k2) {
        const int kb = k2 / 4, ko = (k2 % 4) * 32;
        mma_bf16(tS, sw128_desc(smem_u32(sl + SM::A0 + kb * kTB) + ko, 16, 1024),
                 sw128_desc(smem_u32(sl + SM::B0 + kb * kTB) + ko, 16, 1024), IDESC_S, k2 > 0);
        mma_bf16(tP, sw128_desc(smem_u32(sl + SM::A1 + kb * kTB) + ko, 16, 1024),
                 sw128_desc(smem_u32(sl + SM::B1 + kb * kTB) + ko, 16, 1024), IDESC_S, k2 > 0);
      }
      mma_commit(barS);
    }
    pendS = true;
    ok = mbar_wait(barS, nS & 1);
    if (__syncthreads_or(!ok)) { bad = true; break; }
    ++nS;
    pendS = false;
    tc_fence_after();
    if (last) {  // the own-block operands are consumed: their region takes the residual tiles
      if (tid == 0) load_res(sl, dc.x, cur.h);
      pendR = true;
    }

    // ---- p and ds of row r, columns [32 cc, 32 cc + 32) -> bf16 operand tiles
    {
      const uint32_t* sMask = reinterpret_cast<const uint32_t*>(sl + SM::MASK);
      uint8_t* wds = smem + (COL ? SM::W1 : SM::W0);
      uint8_t* wp = smem + SM::W0;
      float sv[32], dv[32];
      tmem_ld32(tS + lane_off + cc * 32, sv);
      tmem_ld32(tP + lane_off + cc * 32, dv);
      tmem_wait_ld();
      const uint32_t mw = sMask[r * 4 + cc];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float L[8], Dl[8];
        if constexpr (COL) {  // statistics of the 8 destination columns
          const float4* l4 = reinterpret_cast<const float4*>(sL + cc * 32 + q * 8);
          const float4* d4 = reinterpret_cast<const float4*>(sDl + cc * 32 + q * 8);
          const float4 la = l4[0], lb = l4[1], da = d4[0], db = d4[1];
          L[0] = la.x; L[1] = la.y; L[2] = la.z; L[3] = la.w;
          L[4] = lb.x; L[5] = lb.y; L[6] = lb.z; L[7] = lb.w;
          Dl[0] = da.x; Dl[1] = da.y; Dl[2] = da.z; Dl[3] = da.w;
          Dl[4] = db.x; Dl[5] = db.y; Dl[6] = db.z; Dl[7] = db.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            L[e] = lse2;
            Dl[e] = dl;
          }
        }
        uint32_t wd[4], wq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = q * 8 + 2 * e, j1 = j0 + 1;
          const float p0 = ((mw >> j0) & 1u) ? ex2(fmaf(sv[j0], p.qmul, -L[2 * e])) : 0.f;
          const float p1 = ((mw >> j1) & 1u) ? ex2(fmaf(sv[j1], p.qmul, -L[2 * e + 1])) : 0.f;
          wd[e] = bf16x2_bits(p0 * (dv[j0] - Dl[2 * e]), p1 * (dv[j1] - Dl[2 * e + 1]));
          if (COL) wq[e] = bf16x2_bits(p0, p1);
        }
        // 8-column piece c8 of the row: tile c8 / 8, swizzled 16-byte chunk (c8 % 8) ^ (row % 8)
        const int c8 = cc * 4 + q;
        const int off = (c8 / 8) * kTB + r * 128 + (((c8 % 8) ^ (r & 7)) * 16);
        *reinterpret_cast<uint4*>(wds + off) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        if (COL) *reinterpret_cast<uint4*>(wp + off) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
      }
    }
    fence_proxy_async();  // generic stores of the operand tiles -> visible to the tensor cores
    tc_fence_before();
    __syncthreads();

    // ---- gradient products (K = the 128 columns of the tile)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k2 = 0; k2 < kT / 16; ++k2) {
        const uint32_t acc = (!first || k2 > 0) ? 1u : 0u;
        const int aoff = (k2 / 4) * kTB + (k2 % 4) * 32;
        const uint64_t a0 = sw128_desc(smem_u32(smem + SM::W0 + aoff), 16, 1024);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
          // other-block operand, MN-major: 16 rows (K) = two 1024-byte swizzle atoms per step
          const int boff = kb * kTB + k2 * 2048;
          if (!COL) {
            mma_bf16(tG + kb * 64, a0, sw128_desc(smem_u32(sl + SM::B0 + boff), 1024, 1024),
                     IDESC_G, acc);                                     // dQ += dS K
          } else {
            mma_bf16(tG + kb * 64, a0, sw128_desc(smem_u32(sl + SM::B1 + boff), 1024, 1024),
                     IDESC_G, acc);                                     // dV += P^T dO
          }
        }
        if (COL) {
          const uint64_t a1 = sw128_desc(smem_u32(smem + SM::W1 + aoff), 16, 1024);
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
            mma_bf16(tG2 + kb * 64, a1,
                     sw128_desc(smem_u32(sl + SM::B0 + kb * kTB + k2 * 2048), 1024, 1024), IDESC_G,
                     acc);                                              // dK += dS^T Q
        }
      }
      mma_commit(barD);
    }
    pendD = true;
    ok = mbar_wait(barD, nD & 1);
    if (__syncthreads_or(!ok)) { bad = true; break; }
    ++nD;
    pendD = false;
    tc_fence_after();

    if (last) {  // ---- epilogue: residual + this (block, head)'s sums, out by TMA
      ok = mbar_wait(barR, nR & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
      ++nR;
      pendR = false;
      epilogue(sl);
      fence_proxy_async();  // generic stores of the sums -> visible to the TMA stores
      tc_fence_before();
      __syncthreads();
      if (tid == 0) store_res(sl, dc.x, cur.h);
    }
    if constexpr (NS == 1) {
      if (more) {
        if (tid == 0) {  // the slot is free once the products are done and the stores have read it
          bulk_wait_read();
          issue(nx, dn, 0);
        }
        pendL |= 1u;
      }
    }
    cur = nx;
    dc = dn;
    nx = n2;
    dn = d2;
  }

  if (bad && tid == 0) {
    atomicOr(p.err, 2);
    // drain what this block issued (bounded), then free the TMEM
#pragma unroll
    for (int s = 0; s < NS; ++s)
      if ((pendL >> s) & 1u) mbar_wait(barL + s, (phL >> s) & 1u);
    if (pendS) mbar_wait(barS, nS & 1);
    if (pendD) mbar_wait(barD, nD & 1);
    if (pendR) mbar_wait(barR, nR & 1);
  }
  if (tid == 0) bulk_wait();  // the epilogues' stores have completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kCols)
                 : "memory");
}

gattn_status launch_tile_bwd(const TileBwdParams& p, int D, bool col, int num_sms,
                             cudaStream_t st) {
  if (p.n_grp <= 0) return GATTN_OK;
  if (D != 64 && D != 128) {
    set_error("the dense-tile backward supports D = 64 or 128 (got %d)", D);
    return GATTN_ERR_UNSUPPORTED;
  }
  const unsigned grid = (unsigned)(p.n_grp < num_sms ? p.n_grp : num_sms);
  auto go = [&](auto kern, int bytes) -> gattn_status {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
      set_error("tile backward attribute: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    kern<<<grid, kThr, bytes, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("tile backward launch: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    return GATTN_OK;
  };
  if (D == 64)
    return col ? go(tile_bwd_kernel<64, 2, true>, BwdSmem<64, 2, true>::BYTES)
               : go(tile_bwd_kernel<64, 2, false>, BwdSmem<64, 2, false>::BYTES);
  return col ? go(tile_bwd_kernel<128, 1, true>, BwdSmem<128, 1, true>::BYTES)
             : go(tile_bwd_kernel<128, 1, false>, BwdSmem<128, 1, false>::BYTES);
}

}  // namespace gattn
