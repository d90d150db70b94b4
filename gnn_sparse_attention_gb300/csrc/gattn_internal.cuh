// gattn_internal.cuh -- the plan struct and small device helpers shared by
// the translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "gattn.h"

namespace gattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kWarpsPerBlock = 8;
constexpr int kThreads = kWarpsPerBlock * 32;

// ---------------------------------------------------------------------------
// plan (host struct; all arrays are device pointers owned by the plan)
// ---------------------------------------------------------------------------
struct Plan {
  int32_t N = 0;
  int64_t M = 0;
  int32_t T = 256, C = 256;
  int64_t n_light = 0, n_heavy = 0, n_chunks = 0;
  int64_t n_light_src = 0, n_heavy_src = 0, n_src_chunks = 0;
  int32_t max_deg = 0, max_outdeg = 0;
  size_t device_bytes = 0;
  int device = 0;
  int num_sms = 0;
  // CSR side
  int32_t* indptr = nullptr;   // [N+1] copy
  int32_t* indices = nullptr;  // [M] copy
  int32_t* deg = nullptr;      // [N]
  int32_t* hist = nullptr;     // [33]
  int32_t* light = nullptr;    // [N] capacity
  int4* items = nullptr;       // [n_chunks + n_light]: chunks first (w = heavy id), then light (w = -1)
  int32_t* hfirst = nullptr;   // [n_heavy + 1] first chunk (item index) of each heavy node
  int4* sorted = nullptr;      // items by decreasing edge count: (node, e0, e1, item index)
  // merge tree of the heavy chunks: slots [0, n_chunks) are the chunks,
  // slots [n_chunks, n_chunks + n_inner) the inner nodes of every heavy
  // node's tree; parent[s] = -1 at a root
  int32_t* parent = nullptr;   // [n_chunks + n_inner]
  int2* kids = nullptr;        // [n_inner]: (first child slot, child count)
  int64_t n_inner = 0;
  // CSC side
  int32_t* indptrT = nullptr;  // [N+1]
  int32_t* csc_dst = nullptr;  // [M]
  int32_t* csc_eid = nullptr;  // [M]
  int32_t* outdeg = nullptr;   // [N]
  int32_t* hist_out = nullptr; // [33]
  int32_t* light_src = nullptr;
  int4* items_src = nullptr;
  int32_t* hfirst_src = nullptr;
  int4* sorted_src = nullptr;
  int32_t* parent_src = nullptr;
  int2* kids_src = nullptr;
  int64_t n_inner_src = 0;
  // dense-tile path (tile_enable): nodes are cut into blocks of kTileRows
  // ids; a (row block, column block) pair holding at least tile_min edges is
  // a tile, listed in (row block, column block) order with its bit mask
  // (bit j % 128 of row i % 128: 4 words a row).  Edges outside the tiles
  // (and repeated pairs inside them) form the residual CSR, which has its
  // own forward split.
  int32_t tile_min = 0;
  int64_t n_tiles = 0, n_trows = 0, M_res = 0;
  int32_t* tile_rb = nullptr;     // [n_tiles]
  int32_t* tile_cb = nullptr;     // [n_tiles]
  uint32_t* tile_mask = nullptr;  // [n_tiles][128][4]
  int32_t* trow_rb = nullptr;     // [n_trows] row blocks that have tiles
  int32_t* trow_ptr = nullptr;    // [n_trows + 1] their tiles: [trow_ptr[r], trow_ptr[r+1])
  int32_t* indptr_r = nullptr;    // [N+1] residual CSR
  int32_t* indices_r = nullptr;   // [M_res]
  int32_t* res_eid = nullptr;     // [M_res] CSR edge id of each residual edge
  int32_t* tile_slot = nullptr;   // [M] t*16384 + (i%128)*128 + j%128 for tile edges, else -1
                                  // (weighted tiles need n_tiles * 16384 < 2^31)
  int64_t n_light_r = 0, n_chunks_r = 0, n_inner_r = 0;
  int4* items_r = nullptr;
  int4* sorted_r = nullptr;
  int32_t* parent_r = nullptr;
  int2* kids_r = nullptr;
  int32_t* cnt_fwd_r = nullptr;   // [n_inner_r]
  int32_t* cnt_dq_r = nullptr;    // [n_inner_r]
  // backward of a tiled plan: tiles by column block (transposed masks: bit
  // i % 128 of column j % 128, 4 words a column) and the residual CSC with
  // its own source split
  int64_t n_tcols = 0;
  int32_t* tcol_cb = nullptr;       // [n_tcols] column blocks that have tiles
  int32_t* tcol_ptr = nullptr;      // [n_tcols + 1] their tiles in tcol_tile
  int32_t* tcol_tile = nullptr;     // [n_tiles] tile ids by (column block, row block)
  uint32_t* tile_mask_t = nullptr;  // [n_tiles][128][4]
  // step descriptors of the tile backward, per position of the row-order
  // (tile) list and of the column-order list: (own block, other block,
  // tile id, 1 = first / 2 = last tile of its own block)
  int4* tdesc_row = nullptr;        // [n_tiles]
  int4* tdesc_col = nullptr;        // [n_tiles]
  int32_t* indptrT_r = nullptr;     // [N+1]
  int32_t* csc_dst_r = nullptr;     // [M_res] destination of each residual CSC position
  int64_t n_light_src_r = 0, n_chunks_src_r = 0, n_inner_src_r = 0;
  int4* items_src_r = nullptr;
  int4* sorted_src_r = nullptr;
  int32_t* parent_src_r = nullptr;
  int2* kids_src_r = nullptr;
  int32_t* cnt_dkv_r = nullptr;     // [n_inner_src_r]
  // last-arriver counters (zero between calls; the merging warp resets them)
  int32_t* cnt_fwd = nullptr;  // [n_inner]
  int32_t* cnt_dq = nullptr;   // [n_inner]
  int32_t* cnt_dkv = nullptr;  // [n_inner_src]
  int32_t* cnt_da = nullptr;   // [1]
  int32_t* err = nullptr;      // [1] nonzero once a kernel's bounded wait gave up
  int32_t fail_first_wait = 0; // gattn_plan_set_wait_test: attention passes fail their first wait
  std::vector<void*> allocs;   // every device buffer above, freed by destroy
};

constexpr int kMaxBlocksPerSm = 32;  // grid cap of the persistent kernels (bounds da partials)

constexpr int kMaxItemEdges = 256;  // largest heavy threshold and chunk
constexpr int kTreeFanIn = 16;  // children per inner node of a chunk merge tree
constexpr int kTileRows = 128;  // nodes per side of a dense tile

// ---------------------------------------------------------------------------
// math helpers (hardware approximations, fp32)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// ---------------------------------------------------------------------------
// host-side helpers shared by the translation units
// ---------------------------------------------------------------------------
void set_error(const char* fmt, ...);
int grid_for(const Plan& p, int64_t n_items, int blocks_per_sm);

}  // namespace gattn

// The opaque handle of include/gattn.h.
struct gattn_plan {
  gattn::Plan p;
};
