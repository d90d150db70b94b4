// attn_tile.cuh -- parameters of the dense-tile forward (attn_tile.cu).
#pragma once

#include <cuda.h>

#include "gattn_internal.cuh"

namespace gattn {

struct TileParams {
  CUtensorMap mq, mk, mv;      // Q, K, V as [N, H*D] bf16 with 64 x 128 boxes, 128-byte swizzle
  const uint32_t* mask;        // [n_tiles][128][4] tile bit masks
  const int32_t* tile_cb;      // [n_tiles] column block of each tile
  const int32_t* trow_rb;      // [n_trows] row block of each CTA
  const int32_t* trow_ptr;     // [n_trows + 1] tiles of each row block
  int64_t n_trows;
  int N, H;
  float qmul;                  // scale * log2(e)
  void* out;                   // bf16 [N, H, D]: residual result in, merged result out
  float* lse;                  // [N, H]: residual lse in, merged lse out
  int32_t* err;
};

// Tensor map of a [rows, width] bf16 matrix read in 64-column x 128-row
// boxes with the 128-byte swizzle (the tensor cores' operand layout).
bool encode_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t width);

// Launch the dense-tile forward (D = 64 or 128) after the residual pass.
gattn_status launch_tile_fwd(const TileParams& p, int D, cudaStream_t st);

}  // namespace gattn
