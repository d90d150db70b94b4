// attn_tile.cu -- dense-tile forward on the tensor cores (tcgen05 + TMEM).
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", attention-based layers, tensor-core
// optimisation: locally dense neighbourhoods are packed into block tiles so
// that their scores and their weighted sum of values become small dense
// matrix products on the tensor cores; the pages note this pays off on
// locally dense graphs.
//
// The plan cuts the nodes into blocks of 128 ids and keeps every (row block,
// column block) pair with enough edges as a tile with a 128 x 128 bit mask.
// A step is (row block, head h, one of the row block's tiles):
//   TMA (128-byte swizzle) : Q[rows, h], K[cols, h], V[cols, h] as 128 x D
//                            bf16 tiles, and the tile's mask;
//   tcgen05.mma            : S = Q K^T (M = N = 128, K = D) into TMEM;
//   threads                : TMEM lane r is destination row r; 16 warps
//                            split each row's 128 columns into four 32-column
//                            chunks (a warp reads only its own lane quarter).
//                            A thread takes its chunk's masked maximum, the
//                            four chunk maxima of the row meet in shared
//                            memory, and the row's running maximum (base 2)
//                            moves to the largest; the thread writes
//                            p = 2^(s - m) as bf16 into the swizzled P tile
//                            and keeps its chunk's share of the running sum;
//                            when the maximum moved, O's row is rescaled in
//                            TMEM;
//   tcgen05.mma            : O += P V (M = 128, N = D, K = 128) in TMEM.
// After the row block's last tile of head h, the row's sum is assembled from
// the four chunk shares and merged with the residual CSR pass (which ran
// first and wrote out / lse over the edges outside the tiles):
// lse = log(e^lse_t + e^lse_r), out = the two halves weighted by their share
// of the softmax mass.  The residual out tile arrives by TMA in the step's
// Q region (consumed once S is done), the merged rows are written back
// there and leave by a TMA store.  The MMA multiplies the weights rounded to
// bf16 while the normaliser (and so lse, which the backward reuses) sums
// them in fp32, as in FlashAttention.
//
// Schedule: one CTA per SM walks its row blocks (grid stride), the heads
// and the tiles; with two operand slots (D = 64; the kernel also takes three)
// the next step's loads are in flight while the current one computes (one
// slot for D = 128); step descriptors from the plan are loaded two steps
// ahead.  Every mbarrier wait is bounded; a wait that
// gives up is reported through the plan's error word, the block drains what
// it issued (again bounded), frees its TMEM and returns.
#include <cuda.h>

#include "attn_pipe.cuh"
#include "attn_tile.cuh"
#include "tcgen05.cuh"

namespace gattn {

namespace {

constexpr int kT = kTileRows;        // rows / columns of a tile
constexpr int kWarps = 16;           // four warps per TMEM lane quarter
constexpr int kThr = kWarps * 32;    // thread (row r, chunk c): columns [32c, 32c + 32) of row r
constexpr int kTB = kT * 128;        // one 128 x 64 bf16 operand tile (16 KB)
constexpr int kMaskB = kT * 16;      // 128 rows x 4 mask words
constexpr uint32_t kCols = 256;      // TMEM: S [0, 128), O [128, 128 + D)

template <int D, int NS>
struct FwdSmem {
  static constexpr int KB = D / 64;                 // 64-column pieces of a head
  static constexpr int Q = 0;                       // [KB][128 rows][128 B]; the out tile at the end
  static constexpr int K = KB * kTB;
  static constexpr int V = 2 * KB * kTB;
  static constexpr int MASK = 3 * KB * kTB;
  static constexpr int SLOT = MASK + kMaskB;
  static constexpr int P = NS * SLOT;               // P tile: [2][128 rows][128 B]
  static constexpr int RED = P + 2 * kTB;           // [4 chunks][128 rows] fp32 maxima / sums
  static constexpr int BAR = RED + 4 * kT * 4;       // NS + 3 barriers, then the TMEM address
  static constexpr int END = BAR + 8 * (NS + 3) + 8;
  static constexpr int BYTES = END + 1024;          // slack to align the base to 1024
  static_assert(SLOT % 1024 == 0 && P % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
  static_assert(BYTES <= 227 * 1024, "shared memory of one CTA");
};

}  // namespace

template <int D, int NS>
__global__ void __launch_bounds__(kThr, 1) tile_fwd_kernel(const __grid_constant__ TileParams p) {
  using namespace tc;
  using SM = FwdSmem<D, NS>;
  constexpr int KB = SM::KB;
  constexpr uint32_t IDESC_S = f16_idesc(kT, kT, false);
  constexpr uint32_t IDESC_O = f16_idesc(kT, 64, true);  // one 64-column piece of O
  constexpr uint32_t LOAD_BYTES = 3 * KB * kTB + kMaskB;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base: the 128-byte swizzle pattern is a function of
  // the address bits, so every operand tile starts on such a boundary
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sP = smem + SM::P;
  float* sRed = reinterpret_cast<float*>(smem + SM::RED);
  uint64_t* barL = reinterpret_cast<uint64_t*>(smem + SM::BAR);  // [NS] operand slots
  uint64_t* barS = barL + NS;
  uint64_t* barO = barL + NS + 1;
  uint64_t* barR = barL + NS + 2;  // residual out tile of the epilogue
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(barL + NS + 3);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = (warp & 3) * 32 + (tid & 31);  // row of the block = TMEM lane
  const int cc = warp >> 2;                    // 32-column chunk of the row
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(barL + s, 1);
    mbar_init(barS, 1);
    mbar_init(barO, 1);
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
  const uint32_t tS = tmem, tO = tmem + kT;
  const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter

  // TMA loads of one step (descriptor d) into slot s (thread 0)
  auto issue = [&](const TileStep& c, int4 d, int s) {
    uint8_t* sl = smem + s * SM::SLOT;
    fence_proxy_async();
    mbar_expect_tx(barL + s, LOAD_BYTES);
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const int x = c.h * D + kb * 64;
      tma_tile2d(sl + SM::Q + kb * kTB, &p.mq, x, d.x * kT, barL + s);
      tma_tile2d(sl + SM::K + kb * kTB, &p.mk, x, d.y * kT, barL + s);
      tma_tile2d(sl + SM::V + kb * kTB, &p.mv, x, d.y * kT, barL + s);
    }
    bulk_g2s(sl + SM::MASK, p.mask + int64_t(d.z) * kT * 4, kMaskB, barL + s);
  };

  uint32_t phL = 0, pendL = 0, nS = 0, nO = 0, nR = 0;  // barrier phases, loads in flight
  bool pendS = false, pendO = false, pendR = false;
  bool bad = false;

  TileStep cur{-1, 0, 0, 0, -1}, nx{-1, 0, 0, 0, -1};
  int4 dc = make_int4(0, 0, 0, 0), dn = make_int4(0, 0, 0, 0);
  if (blockIdx.x < p.n_grp) {
    cur = tile_step_block(p, blockIdx.x, p.grp_ptr[blockIdx.x]);
    dc = p.desc[cur.q];
    nx = tile_step_after(p, cur, dc);
    if (nx.g >= 0) dn = p.desc[nx.q];
    if (tid == 0) issue(cur, dc, 0);
    pendL = 1u;
    if constexpr (NS == 3) {  // three slots: loads run two steps ahead
      if (nx.g >= 0) {
        if (tid == 0) issue(nx, dn, 1);
        pendL |= 2u;
      }
    }
  }
  float m = neg_inf(), l = 0.f;  // the row's running maximum (base 2) and this chunk's share of its sum
  for (int k = 0; cur.g >= 0; ++k) {
    const int s = k % NS;
    const bool more = nx.g >= 0;
    const TileStep n2 = more ? tile_step_after(p, nx, dn) : TileStep{-1, 0, 0, 0, -1};
    const int4 d2 = n2.g >= 0 ? p.desc[n2.q] : make_int4(0, 0, 0, 0);  // used next step
    const bool first = dc.w & 1;
    const bool last = dc.w & 2;
    if constexpr (NS == 2) {
      if (more) {
        // slot s ^ 1 was released by the previous step once its epilogue's
        // store has read the out tile
        if (tid == 0) {
          bulk_wait_read();
          issue(nx, dn, s ^ 1);
        }
        pendL |= 1u << (s ^ 1);
      }
    } else if constexpr (NS == 3) {
      if (n2.g >= 0) {
        // slot (k + 2) % 3 held the previous step, released the same way
        const int s2 = (k + 2) % 3;
        if (tid == 0) {
          bulk_wait_read();
          issue(n2, d2, s2);
        }
        pendL |= 1u << s2;
      }
    }
    const int node = dc.x * kT + r;
    const int64_t srow = int64_t(node) * p.H + cur.h;
    float lres = neg_inf();  // the residual pass's lse of the row (used by the epilogue)
    if (last && node < p.N) lres = p.lse[srow];
    if (first) {
      m = neg_inf();
      l = 0.f;
    }
    bool ok = mbar_wait(barL + s, (phL >> s) & 1u);
    if (__syncthreads_or(!ok)) { bad = true; break; }
    phL ^= 1u << s;
    pendL &= ~(1u << s);

    // ---- S = Q K^T
    uint8_t* sl = smem + s * SM::SLOT;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k2 = 0; k2 < D / 16; ++k2) {
        const int kb = k2 / 4, ko = (k2 % 4) * 32;
        mma_bf16(tS, sw128_desc(smem_u32(sl + SM::Q + kb * kTB) + ko, 16, 1024),
                 sw128_desc(smem_u32(sl + SM::K + kb * kTB) + ko, 16, 1024), IDESC_S, k2 > 0);
      }
      mma_commit(barS);
    }
    pendS = true;
    ok = mbar_wait(barS, nS & 1);
    if (__syncthreads_or(!ok)) { bad = true; break; }
    ++nS;
    pendS = false;
    tc_fence_after();
    if (last) {  // Q is consumed: its region takes the residual out tile
      if (tid == 0) {
        fence_proxy_async();
        mbar_expect_tx(barR, KB * kTB);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
          tma_tile2d(sl + SM::Q + kb * kTB, &p.mo, cur.h * D + kb * 64, dc.x * kT, barR);
      }
      pendR = true;
    }

    // ---- online softmax of row r over columns [32 cc, 32 cc + 32)
    float sv[32];
    tmem_ld32(tS + lane_off + cc * 32, sv);
    tmem_wait_ld();
    const uint32_t mw = reinterpret_cast<const uint32_t*>(sl + SM::MASK)[r * 4 + cc];
    float cm = neg_inf();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      sv[j] *= p.qmul;
      if ((mw >> j) & 1u) cm = fmaxf(cm, sv[j]);
    }
    sRed[cc * kT + r] = cm;
    __syncthreads();  // the four chunk maxima of every row
    float mx = m;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) mx = fmaxf(mx, sRed[c4 * kT + r]);
    const float base = mx == neg_inf() ? 0.f : mx;
    const float corr = ex2(m - base);
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j0 = q * 8 + 2 * e, j1 = j0 + 1;
        const float p0 = ((mw >> j0) & 1u) ? ex2(sv[j0] - base) : 0.f;
        const float p1 = ((mw >> j1) & 1u) ? ex2(sv[j1] - base) : 0.f;
        w[e] = bf16x2_bits(p0, p1);
        sum += p0 + p1;
      }
      // 8-column piece c8 of the row: tile c8 / 8, swizzled 16-byte chunk (c8 % 8) ^ (row % 8)
      const int c8 = cc * 4 + q;
      *reinterpret_cast<uint4*>(sP + (c8 / 8) * kTB + r * 128 + (((c8 % 8) ^ (r & 7)) * 16)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    l = l * corr + sum;
    m = mx;
    // rescale O's row when the running maximum moved (chunk threads cc < D / 32
    // own O's 32-column pieces; the condition is uniform within a warp's use)
    if (!first && cc < D / 32 && __any_sync(FULL, corr != 1.f)) {
      float o[32];
      tmem_ld32(tO + lane_off + cc * 32, o);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] *= corr;
      tmem_st32(tO + lane_off + cc * 32, o);
      tmem_wait_st();
    }
    fence_proxy_async();  // P (generic stores) -> visible to the tensor cores
    tc_fence_before();
    __syncthreads();

    // ---- O += P V
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k2 = 0; k2 < kT / 16; ++k2) {
        const uint64_t a = sw128_desc(smem_u32(sP + (k2 / 4) * kTB) + (k2 % 4) * 32, 16, 1024);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
          // V tile kb: MN-major, 16 rows (K) = two 1024-byte swizzle atoms per step
          const uint64_t b = sw128_desc(smem_u32(sl + SM::V + kb * kTB) + k2 * 2048, 1024, 1024);
          mma_bf16(tO + kb * 64, a, b, IDESC_O, (!first || k2 > 0) ? 1u : 0u);
        }
      }
      mma_commit(barO);
    }
    pendO = true;
    ok = mbar_wait(barO, nO & 1);
    if (__syncthreads_or(!ok)) { bad = true; break; }
    ++nO;
    pendO = false;
    tc_fence_after();

    if (last) {  // ---- epilogue: merge with the residual pass, out by TMA
      sRed[cc * kT + r] = l;  // the maxima were read before the mid-step barrier
      ok = mbar_wait(barR, nR & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
      ++nR;
      pendR = false;
      float lt = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) lt += sRed[c4 * kT + r];
      const float Lt = lt > 0.f ? m + lg2(lt) : neg_inf();  // base 2
      const float Lr = lres * kLog2e;                        // -inf if no residual edge
      const float Lm = fmaxf(Lt, Lr);
      float L = neg_inf(), wt = 0.f, wr = 0.f;
      if (Lm != neg_inf()) {
        L = Lm + lg2(ex2(Lt - Lm) + ex2(Lr - Lm));
        wt = lt > 0.f ? ex2(m - L) : 0.f;  // O is scaled by 2^-m
        wr = ex2(Lr - L);
      }
      if (cc < D / 32) {  // warp-uniform: the TMEM load is a whole-warp instruction
        float o[32];
        tmem_ld32(tO + lane_off + cc * 32, o);
        tmem_wait_ld();
        uint8_t* row = sl + SM::Q + ((cc * 32) / 64) * kTB + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4* ptr = reinterpret_cast<uint4*>(row + (((((cc * 32) % 64) / 8 + q) ^ (r & 7)) * 16));
          const uint4 u = *ptr;
          const uint32_t in[4] = {u.x, u.y, u.z, u.w};
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float r0 = __uint_as_float(in[e] << 16), r1 = __uint_as_float(in[e] & 0xffff0000u);
            w[e] = bf16x2_bits(o[q * 8 + 2 * e] * wt + r0 * wr, o[q * 8 + 2 * e + 1] * wt + r1 * wr);
          }
          *ptr = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (cc == 0 && node < p.N) p.lse[srow] = Lm == neg_inf() ? neg_inf() : L * kLn2;
      fence_proxy_async();  // generic stores of the merged rows -> visible to the TMA store
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
          tma_store2d(&p.mo, cur.h * D + kb * 64, dc.x * kT, sl + SM::Q + kb * kTB);
        bulk_commit();
      }
    }
    if constexpr (NS == 1) {
      if (more) {
        if (tid == 0) {  // the slot is free once O's product is done and the store has read it
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
    if (pendO) mbar_wait(barO, nO & 1);
    if (pendR) mbar_wait(barR, nR & 1);
  }
  if (tid == 0) bulk_wait();  // the epilogues' stores have completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kCols)
                 : "memory");
}

gattn_status launch_tile_fwd(const TileParams& p, int D, int num_sms, cudaStream_t st) {
  if (p.n_grp <= 0) return GATTN_OK;
  if (D != 64 && D != 128) {
    set_error("the dense-tile forward supports D = 64 or 128 (got %d)", D);
    return GATTN_ERR_UNSUPPORTED;
  }
  const unsigned grid = (unsigned)(p.n_grp < num_sms ? p.n_grp : num_sms);
  auto go = [&](auto kern, int bytes) -> gattn_status {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
      set_error("tile kernel attribute: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    kern<<<grid, kThr, bytes, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("tile kernel launch: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    return GATTN_OK;
  };
  // D = 64: two operand slots (three, with the loads of two steps in flight,
  // measured no faster on the block-model graphs and take 50 KB more)
  if (D == 64) return go(tile_fwd_kernel<64, 2>, FwdSmem<64, 2>::BYTES);
  return go(tile_fwd_kernel<128, 1>, FwdSmem<128, 1>::BYTES);
}

}  // namespace gattn
