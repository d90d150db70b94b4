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
// One CTA of 128 threads takes one row block; thread r owns destination row
// r of the block, which is also TMEM lane r of every accumulator.  For each
// head h and each tile of the row block:
//   TMA (128-byte swizzle) : Q[rows, h] (once per head), K[cols, h], V[cols, h]
//                            as 128 x D bf16 tiles, and the tile's mask;
//   tcgen05.mma            : S = Q K^T (M = N = 128, K = D) into TMEM;
//   threads                : row r reads its 128 scores from TMEM, drops the
//                            masked-out columns, updates the running max and
//                            sum (base-2 units) and writes p = 2^(s - m) as
//                            bf16 into the P tile (the same swizzled layout);
//                            when the max grew, O's row is rescaled in TMEM;
//   tcgen05.mma            : O += P V (M = 128, N = D, K = 128) in TMEM.
// After the head's last tile each thread merges its row with the residual
// CSR pass (which ran first and wrote out / lse over the edges outside the
// tiles): lse = log(e^lse_t + e^lse_r), out = the two halves weighted by
// their share of the softmax mass.  The MMA multiplies the weights rounded
// to bf16 while the normaliser (and so lse, which the backward reuses) sums
// them in fp32, as in FlashAttention.
//
// Every mbarrier wait is bounded; a wait that gives up is reported through
// the plan's error word, the block drains what it issued (again bounded),
// frees its TMEM and returns.
#include <cuda.h>

#include "attn_pipe.cuh"
#include "attn_tile.cuh"
#include "tcgen05.cuh"

namespace gattn {

namespace {

constexpr int kT = kTileRows;             // 128 rows / columns per tile
constexpr int kThreadsTile = 128;         // one thread per row
constexpr int kTileBytes = kT * 128;      // one 128 x 64 bf16 operand tile (16 KB)
constexpr int kMaskWords = kT * 4;
constexpr uint32_t kTmemCols = 256;       // S: columns [0, 128), O: [128, 128 + D)

template <int D>
struct TileSmem {
  static constexpr int KB = D / 64;                 // 64-wide K blocks of a head
  static constexpr int Q = 0;                       // [KB][128 rows][128 B]
  static constexpr int K = Q + KB * kTileBytes;
  static constexpr int V = K + KB * kTileBytes;     // [KB][128 rows][128 B]
  static constexpr int P = V + KB * kTileBytes;     // [2][128 rows][128 B]
  static constexpr int MASK = P + 2 * kTileBytes;
  static constexpr int BAR = MASK + kMaskWords * 4;  // load, S, O barriers + TMEM address
  static constexpr int END = BAR + 64;
  static constexpr int BYTES = END + 1024;          // slack to align the base to 1024
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreadsTile) tile_fwd_kernel(const __grid_constant__ TileParams p) {
  using namespace tc;
  using SM = TileSmem<D>;
  constexpr int KB = SM::KB;
  constexpr uint32_t IDESC_S = f16_idesc(kT, kT, false);
  constexpr uint32_t IDESC_O = f16_idesc(kT, 64, true);  // one 64-column half of O
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base: the 128-byte swizzle pattern is a function of
  // the address bits, so every operand tile starts on such a boundary
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + SM::Q;
  uint8_t* sK = smem + SM::K;
  uint8_t* sV = smem + SM::V;
  uint8_t* sP = smem + SM::P;
  const uint32_t* sMask = reinterpret_cast<const uint32_t*>(smem + SM::MASK);
  uint64_t* barLoad = reinterpret_cast<uint64_t*>(smem + SM::BAR);
  uint64_t* barS = barLoad + 1;
  uint64_t* barO = barLoad + 2;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(barLoad + 3);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int rb = p.trow_rb[blockIdx.x];
  const int t0 = p.trow_ptr[blockIdx.x], t1 = p.trow_ptr[blockIdx.x + 1];
  const int node = rb * kT + tid;

  if (tid == 0) {
    mbar_init(barLoad, 1);
    mbar_init(barS, 1);
    mbar_init(barO, 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
            smem_u32(sTmem)),
        "r"(kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem, tO = tmem + kT;
  const uint32_t lane_off = uint32_t(warp * 32) << 16;  // this warp's TMEM lane quarter

  uint32_t nLoad = 0, nS = 0, nO = 0;  // completed phases of each barrier
  bool pendLoad = false, pendS = false, pendO = false;
  bool bad = false;

  for (int h = 0; h < p.H && !bad; ++h) {
    float m = neg_inf(), l = 0.f;  // running max (base 2) and sum of this row
    for (int t = t0; t < t1 && !bad; ++t) {
      // ---- loads (the previous tile's MMAs have completed: barO was waited)
      if (tid == 0) {
        fence_proxy_async();
        const uint32_t bytes =
            (t == t0 ? KB * kTileBytes : 0) + 2 * KB * kTileBytes + kMaskWords * 4;
        mbar_expect_tx(barLoad, bytes);
        const int cb = p.tile_cb[t];
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
          if (t == t0) tma_tile2d(sQ + kb * kTileBytes, &p.mq, h * D + kb * 64, rb * kT, barLoad);
          tma_tile2d(sK + kb * kTileBytes, &p.mk, h * D + kb * 64, cb * kT, barLoad);
          tma_tile2d(sV + kb * kTileBytes, &p.mv, h * D + kb * 64, cb * kT, barLoad);
        }
        bulk_g2s(smem + SM::MASK, p.mask + int64_t(t) * kMaskWords, kMaskWords * 4, barLoad);
      }
      pendLoad = true;
      bool ok = mbar_wait(barLoad, nLoad & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
      ++nLoad;
      pendLoad = false;

      // ---- S = Q K^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const int kb = k / 4, ko = (k % 4) * 32;
          const uint64_t a = sw128_desc(smem_u32(sQ + kb * kTileBytes) + ko, 16, 1024);
          const uint64_t b = sw128_desc(smem_u32(sK + kb * kTileBytes) + ko, 16, 1024);
          mma_bf16(tS, a, b, IDESC_S, k > 0);
        }
        mma_commit(barS);
      }
      pendS = true;
      ok = mbar_wait(barS, nS & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
      ++nS;
      pendS = false;
      tc_fence_after();

      // ---- softmax of row `tid` over the tile's columns
      float s[kT];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, s + c * 32);
      tmem_wait_ld();
      uint32_t mw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) mw[c] = sMask[tid * 4 + c];
      float mx = m;
#pragma unroll
      for (int j = 0; j < kT; ++j) {
        s[j] *= p.qmul;
        if ((mw[j / 32] >> (j % 32)) & 1u) mx = fmaxf(mx, s[j]);
      }
      const float base = mx == neg_inf() ? 0.f : mx;
      const float corr = ex2(m - base);
      float sum = 0.f;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = kb * 64 + ch * 8 + 2 * q;
            const float p0 = ((mw[j / 32] >> (j % 32)) & 1u) ? ex2(s[j] - base) : 0.f;
            const float p1 = ((mw[(j + 1) / 32] >> ((j + 1) % 32)) & 1u) ? ex2(s[j + 1] - base) : 0.f;
            w[q] = bf16x2_bits(p0, p1);
            sum += p0 + p1;
          }
          // K-major 128-byte swizzle: 16-byte chunk ch of row r sits at chunk ch ^ (r % 8)
          uint8_t* dst = sP + kb * kTileBytes + tid * 128 + ((ch ^ (tid & 7)) * 16);
          *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      l = l * corr + sum;
      m = mx;
      // rescale this row of O when the running max moved (warp-uniform TMEM access)
      if (t > t0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(tO + lane_off + c * 32, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async();  // P (generic stores) -> visible to the tensor cores
      tc_fence_before();
      __syncthreads();

      // ---- O += P V
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kT / 16; ++k) {
          const uint64_t a = sw128_desc(smem_u32(sP + (k / 4) * kTileBytes) + (k % 4) * 32, 16, 1024);
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            // V tile kb: MN-major, 16 rows (K) = two 1024-byte swizzle atoms per step
            const uint64_t b = sw128_desc(smem_u32(sV + kb * kTileBytes) + k * 2048, 1024, 1024);
            mma_bf16(tO + kb * 64, a, b, IDESC_O, (t > t0 || k > 0) ? 1u : 0u);
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
    }
    if (bad) break;

    // ---- epilogue: merge with the residual pass and write row `tid`, head h
    float o[D];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + lane_off + c * 32, o + c * 32);
    tmem_wait_ld();
    if (node < p.N) {
      const int64_t row = int64_t(node) * p.H + h;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + row * D;
      const float Lt = l > 0.f ? m + lg2(l) : neg_inf();           // base 2
      const float Lr = p.lse[row] * kLog2e;                        // -inf if no residual edge
      const float Lm = fmaxf(Lt, Lr);
      if (Lm == neg_inf()) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
          reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
        p.lse[row] = neg_inf();
      } else {
        const float L = Lm + lg2(ex2(Lt - Lm) + ex2(Lr - Lm));
        const float wt = l > 0.f ? ex2(m - L) : 0.f;               // O is scaled by 2^-m
        const float wr = ex2(Lr - L);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 u = reinterpret_cast<const uint4*>(orow)[c];
          const uint32_t in[4] = {u.x, u.y, u.z, u.w};
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float r0 = __uint_as_float(in[q] << 16), r1 = __uint_as_float(in[q] & 0xffff0000u);
            w[q] = bf16x2_bits(o[c * 8 + 2 * q] * wt + r0 * wr, o[c * 8 + 2 * q + 1] * wt + r1 * wr);
          }
          reinterpret_cast<uint4*>(orow)[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        p.lse[row] = L * kLn2;
      }
    }
    tc_fence_before();
    __syncthreads();  // every thread is done reading O before the next head overwrites it
    tc_fence_after();
  }

  if (bad) {
    if (tid == 0) atomicOr(p.err, 2);
    // drain what this block issued (bounded), then free the TMEM
    if (tid == 0) {
      if (pendLoad) mbar_wait(barLoad, nLoad & 1);
      if (pendS) mbar_wait(barS, nS & 1);
      if (pendO) mbar_wait(barO, nO & 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

gattn_status launch_tile_fwd(const TileParams& p, int D, cudaStream_t st) {
  if (p.n_trows <= 0) return GATTN_OK;
  if (D != 64 && D != 128) {
    set_error("the dense-tile forward supports D = 64 or 128 (got %d)", D);
    return GATTN_ERR_UNSUPPORTED;
  }
  auto go = [&](auto kern, int bytes) -> gattn_status {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
      set_error("tile kernel attribute: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    kern<<<(unsigned)p.n_trows, kThreadsTile, bytes, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("tile kernel launch: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    return GATTN_OK;
  };
  if (D == 64) return go(tile_fwd_kernel<64>, TileSmem<64>::BYTES);
  return go(tile_fwd_kernel<128>, TileSmem<128>::BYTES);
}

}  // namespace gattn
