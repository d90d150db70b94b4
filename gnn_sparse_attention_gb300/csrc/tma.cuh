// tma.cuh -- tensor maps for row gathers and the tile::gather4 copy.
//
// A dense [N, H, D] tensor is described to the TMA engine as a 2-D tensor of
// N rows of HD elements; one tile::gather4 copy fetches four arbitrary rows
// (by row index) of up to 256 elements each into shared memory, completing
// on an mbarrier.  A row index of N (past the end) is filled with zeros and
// reads nothing, which is how unused slots of a gather are padded.  Per-node
// fp32 statistics (lse, Delta: [N, H]) use the same scheme when their rows are
// whole 16-byte pieces.
#pragma once

#include <cuda.h>

#include "gattn_internal.cuh"

namespace gattn {

constexpr int kGatherBoxMax = 256;  // elements per row piece of one gather

// Host: encode a row-gather map of `rows` rows of `width` elements of
// `elem_bytes` bytes at `base` (row stride width * elem_bytes).  The box is
// one row of min(width, 256) elements.  Returns false (message set) when the
// driver refuses.
bool encode_rows_map(CUtensorMap* map, const void* base, int elem_bytes, bool is_bf16,
                     int64_t rows, int64_t width);

// Device: copy rows r0..r3 (elements [col, col + box) of each) of `map` to
// dst (4 x box elements, row after row), counting bytes on `bar`.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, int col, int r0,
                                            int r1, int r2, int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(
          static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
      : "memory");
}

}  // namespace gattn
