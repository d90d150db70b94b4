// attn_tile.cuh -- parameters of the dense-tile forward (attn_tile.cu).
#pragma once

#include <cuda.h>

#include "gattn_internal.cuh"

namespace gattn {

// Forward of the tiles (attn_tile.cu): one CTA per SM walks the row blocks
// that have tiles, the heads, and each row block's tiles.
struct TileParams {
  CUtensorMap mq, mk, mv;      // Q, K, V as [N, H*D] bf16 with 64 x 128 boxes, 128-byte swizzle
  CUtensorMap mo;              // out, the same way (residual result in, merged result out)
  const uint32_t* mask;        // [n_tiles][128][4] tile bit masks
  const int4* desc;            // [n_tiles] per tile: row block, column block, tile id,
                               // flags (1 first, 2 last tile of its row block)
  const int32_t* grp_ptr;      // [n_grp + 1] tiles of each row block that has tiles
  int64_t n_grp;
  int N, H;
  float qmul;                  // scale * log2(e)
  float* lse;                  // [N, H]: residual lse in, merged lse out
  int32_t* err;
};

// Backward of the tiles (attn_tile_bwd.cu).  The row kernel (COL = false)
// walks the row blocks that have tiles and adds dQ; the column kernel (COL =
// true) walks the column blocks and adds dK, dV.  "Own" rows are the
// block the CTA works on, "other" rows the tile's block on the other side.
struct TileBwdParams {
  CUtensorMap ma0, ma1;        // own block:   row kernel Q, dO;  column kernel K, V
  CUtensorMap mb0, mb1;        // other block: row kernel K, V;   column kernel Q, dO
  CUtensorMap mg1, mg2;        // gradients (tile maps of g1, g2)
  const uint32_t* mask;        // row kernel: tile masks; column kernel: transposed masks
  const int4* desc;            // [n_tiles] per list position: own block, other block, tile
                               // id, flags (1 first, 2 last tile of the own block)
  const int32_t* grp_ptr;      // [n_grp + 1] list positions of each own block's tiles
  int64_t n_grp;
  int N, H;
  float qmul;                  // scale * log2(e)
  float scale;
  const float* lse;            // [N, H]
  const float* delta;          // [N, 2H]: lse * log2(e) of the H heads, then Delta
  void* g1;                    // bf16: row kernel dQ, column kernel dK (residual in, sum out)
  void* g2;                    // bf16: column kernel dV
  int32_t* err;
};

// Launch the row (dQ) or column (dK, dV) tile backward, D = 64 or 128,
// after the residual pass of the same side.
gattn_status launch_tile_bwd(const TileBwdParams& p, int D, bool col, int num_sms, cudaStream_t st);

// A step of the tile kernels: block list entry g, head h, position q in the
// tile list; q0 is the first position of g's tiles and qn that of the
// CTA's next block (-1 past the end), fetched when the block starts.  The
// CTAs take the blocks in grid stride, and for each block every head in
// turn, and for each head the block's tiles.
struct TileStep {
  int g, h, q, q0, qn;
};

template <class P>
__device__ __forceinline__ TileStep tile_step_block(const P& p, int64_t g, int q0) {
  const int64_t gn = g + gridDim.x;
  return TileStep{int(g), 0, q0, q0, gn < p.n_grp ? p.grp_ptr[gn] : -1};
}

// The step after c, whose descriptor is d (no loads but the next block's qn).
template <class P>
__device__ __forceinline__ TileStep tile_step_after(const P& p, const TileStep& c, int4 d) {
  if (!(d.w & 2)) return TileStep{c.g, c.h, c.q + 1, c.q0, c.qn};
  if (c.h + 1 < p.H) return TileStep{c.g, c.h + 1, c.q0, c.q0, c.qn};
  if (c.qn < 0) return TileStep{-1, 0, 0, 0, -1};
  return tile_step_block(p, int64_t(c.g) + gridDim.x, c.qn);
}

// Tensor map of a [rows, width] bf16 matrix read in 64-column x 128-row
// boxes with the 128-byte swizzle (the tensor cores' operand layout).
bool encode_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t width);

// Launch the dense-tile forward (D = 64 or 128) after the residual pass.
gattn_status launch_tile_fwd(const TileParams& p, int D, int num_sms, cudaStream_t st);

}  // namespace gattn
