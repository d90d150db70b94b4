// spmm_tile.cu -- the tensor-core part of the weighted block-sparse (WSB)
// SpMM: for every 128-node row block with dense tiles, y[rows] += sum over
// its tiles W_t x[cols] on tcgen05, added to the residual CSR result.
//
// "On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
// technical summaries, "Methodology", SpMM-based convolutions: a weighted
// block-sparse format packs local neighbourhoods into tiles for the tensor
// cores.  Here a tile is the plan's 128 x 128 block; its bf16 weights (the
// edge weights at their (row, column) slots, zeros elsewhere) form the A
// operand (K-major, the rows' sources contiguous) and the 128 source rows of
// x the B operand (MN-major, features contiguous), both loaded by TMA with
// the 128-byte swizzle; the fp32 product accumulates in TMEM over the row
// block's tiles, 64 feature columns per MMA, up to 256 columns per pass.
// Thread r of the 128-thread CTA owns row r (TMEM lane r) in the epilogue:
// after a pass's last tile the residual y tile comes in by TMA over the
// source-row buffer (free once the products are done), each thread adds its
// row, and the sums leave by a TMA store.
// Every wait is bounded; a failed wait is recorded in the plan's error word
// and the CTA drains (bounded), frees its TMEM and returns.
#include "spmm.cuh"
#include "tcgen05.cuh"

namespace gattn {

namespace {

constexpr int kRows = kTileRows;
constexpr int kBox = kRows * 128;  // one 128 x 64 bf16 tile, 16 KB

template <int FC>
struct WsbSmem {
  static constexpr int W = 0;                  // [2][128][128 B] weight tile (two K blocks)
  static constexpr int X = 2 * kBox;           // [FC / 64][128][128 B] source rows
  static constexpr int BAR = X + (FC / 64) * kBox;
  static constexpr int BYTES = BAR + 64 + 1024;
};

template <int FC>
__global__ void __launch_bounds__(128) wsb_tile_kernel(const __grid_constant__ WsbParams p) {
  using namespace tc;
  using SM = WsbSmem<FC>;
  constexpr uint32_t IDESC = f16_idesc(kRows, 64, true);
  constexpr uint32_t COLS = FC < 32 ? 32 : FC;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sW = smem + SM::W;
  uint8_t* sX = smem + SM::X;
  uint64_t* barLoad = reinterpret_cast<uint64_t*>(smem + SM::BAR);
  uint64_t* barMma = barLoad + 1;
  uint64_t* barY = barLoad + 2;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(barLoad + 3);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int rb = p.trow_rb[blockIdx.x];
  const int t0 = p.trow_ptr[blockIdx.x], t1 = p.trow_ptr[blockIdx.x + 1];
  if (tid == 0) {
    mbar_init(barLoad, 1);
    mbar_init(barMma, 1);
    mbar_init(barY, 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(sTmem)),
                 "r"(COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tD = *sTmem;
  const uint32_t lane_off = uint32_t(warp * 32) << 16;
  uint32_t nLoad = 0, nMma = 0, nY = 0;
  bool pendLoad = false, pendMma = false, pendY = false, bad = false;

  for (int f0 = 0; f0 < p.F && !bad; f0 += FC) {
    for (int t = t0; t < t1 && !bad; ++t) {
      if (tid == 0) {
        bulk_wait_read();  // the previous pass's y store has read the source-row buffer
        fence_proxy_async();
        mbar_expect_tx(barLoad, 2 * kBox + (FC / 64) * kBox);
        const int cb = p.tile_cb[t];
        tma_tile2d(sW, &p.mw, 0, t * kRows, barLoad);
        tma_tile2d(sW + kBox, &p.mw, 64, t * kRows, barLoad);
#pragma unroll
        for (int n = 0; n < FC / 64; ++n)
          tma_tile2d(sX + n * kBox, &p.mx, f0 + n * 64, cb * kRows, barLoad);
      }
      pendLoad = true;
      bool ok = mbar_wait(barLoad, nLoad & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
      ++nLoad;
      pendLoad = false;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kRows / 16; ++k) {
          const uint64_t a = sw128_desc(smem_u32(sW + (k / 4) * kBox) + (k % 4) * 32, 16, 1024);
#pragma unroll
          for (int n = 0; n < FC / 64; ++n) {
            const uint64_t b = sw128_desc(smem_u32(sX + n * kBox) + k * 2048, 1024, 1024);
            mma_bf16(tD + n * 64, a, b, IDESC, (t > t0 || k > 0) ? 1u : 0u);
          }
        }
        mma_commit(barMma);
      }
      pendMma = true;
      ok = mbar_wait(barMma, nMma & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
      ++nMma;
      pendMma = false;
      tc_fence_after();
    }
    if (bad) break;
    // epilogue: y[rows][f0 .. f0 + FC) += D, the y tile through the
    // source-row buffer (64-column boxes, 128-byte swizzle)
    if (tid == 0) {
      fence_proxy_async();
      mbar_expect_tx(barY, (FC / 64) * kBox);
#pragma unroll
      for (int n = 0; n < FC / 64; ++n) tma_tile2d(sX + n * kBox, &p.my, f0 + n * 64, rb * kRows, barY);
    }
    pendY = true;
    {
      const bool ok = mbar_wait(barY, nY & 1);
      if (__syncthreads_or(!ok)) { bad = true; break; }
    }
    ++nY;
    pendY = false;
#pragma unroll
    for (int c = 0; c < FC / 32; ++c) {
      float d[32];
      tmem_ld32(tD + lane_off + c * 32, d);
      tmem_wait_ld();
      uint8_t* row = sX + (c / 2) * kBox + tid * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4* ptr = reinterpret_cast<uint4*>(row + ((((c % 2) * 4 + q) ^ (tid & 7)) * 16));
        const uint4 u = *ptr;
        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float lo = __uint_as_float(in[h] << 16) + d[q * 8 + 2 * h];
          const float hi = __uint_as_float(in[h] & 0xffff0000u) + d[q * 8 + 2 * h + 1];
          w[h] = bf16x2_bits(lo, hi);
        }
        *ptr = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async();  // generic stores of the sums -> visible to the TMA store
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
#pragma unroll
      for (int n = 0; n < FC / 64; ++n) tma_store2d(&p.my, f0 + n * 64, rb * kRows, sX + n * kBox);
      bulk_commit();
    }
    tc_fence_before();
    __syncthreads();  // D is read out before the next column pass overwrites it
    tc_fence_after();
  }

  if (bad && tid == 0) {
    atomicOr(p.err, 4);
    if (pendLoad) mbar_wait(barLoad, nLoad & 1);
    if (pendMma) mbar_wait(barMma, nMma & 1);
    if (pendY) mbar_wait(barY, nY & 1);
  }
  if (tid == 0) bulk_wait();  // the y stores have completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tD), "r"(COLS)
                 : "memory");
}

}  // namespace

gattn_status launch_wsb_tiles(const WsbParams& p, cudaStream_t st) {
  if (p.n_trows <= 0) return GATTN_OK;
  auto go = [&](auto kern, int bytes) -> gattn_status {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
      kern<<<(unsigned)p.n_trows, 128, bytes, st>>>(p);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
      set_error("WSB tile kernel launch: %s", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    return GATTN_OK;
  };
  if (p.F % 256 == 0) return go(wsb_tile_kernel<256>, WsbSmem<256>::BYTES);
  if (p.F % 128 == 0) return go(wsb_tile_kernel<128>, WsbSmem<128>::BYTES);
  if (p.F % 64 == 0) return go(wsb_tile_kernel<64>, WsbSmem<64>::BYTES);
  set_error("WSB tiles need F a multiple of 64 (got %d)", p.F);
  return GATTN_ERR_UNSUPPORTED;
}

}  // namespace gattn
