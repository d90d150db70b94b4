// gattn_internal.cuh -- shared device helpers, lane layout and the plan struct.
//
// Row layout used by every attention kernel.  A row of a dense tensor is the
// H*D values of one node, RB = H*D*sizeof(T) bytes.  It is cut into 16-byte
// chunks (VEC = 16/sizeof(T) elements).  A warp works on one destination (or
// one edge chunk of it) at a time; LPR lanes cover a row, so EPW = 32/LPR
// edges are in flight per warp step (the warp's "slots"), and each lane holds
// CPL chunks of the row (CPL > 1 only when a row exceeds 512 bytes).  The
// lanes of one head (LPH = D/VEC of them, consecutive) combine their partial
// dot products with butterfly shuffles.
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
  int4* units = nullptr;       // [n_units]: (item_begin, item_end, edge_begin, edge_end)
  int64_t n_units = 0;
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
  int4* units_src = nullptr;
  int64_t n_units_src = 0;
  int4* sorted_src = nullptr;
  int32_t* parent_src = nullptr;
  int2* kids_src = nullptr;
  int64_t n_inner_src = 0;
  // last-arriver counters (zero between calls; the merging warp resets them)
  int32_t* cnt_fwd = nullptr;  // [n_inner]
  int32_t* cnt_dq = nullptr;   // [n_inner]
  int32_t* cnt_dkv = nullptr;  // [n_inner_src]
  int32_t* cnt_da = nullptr;   // [1]
  int32_t* err = nullptr;      // [1] nonzero once a kernel's bounded wait gave up
  std::vector<void*> allocs;   // every device buffer above, freed by destroy
};

constexpr int kMaxBlocksPerSm = 32;  // grid cap of the persistent kernels (bounds da partials)

// Work units: runs of consecutive items whose edges are contiguous, at most
// kUnitItems items, all starting inside one kUnitBucket-edge bucket of the
// item list's edge prefix.  With items of at most kMaxItemEdges edges a unit
// spans at most kUnitEdges edges.
constexpr int kUnitItems = 32;
constexpr int kUnitBucket = 128;
constexpr int kMaxItemEdges = 256;
constexpr int kUnitEdges = kUnitBucket + kMaxItemEdges;
constexpr int kTreeFanIn = 16;  // children per inner node of a chunk merge tree

// ---------------------------------------------------------------------------
// lane layout
// ---------------------------------------------------------------------------
template <typename T, int RB>
struct Layout {
  static constexpr int VEC = 16 / (int)sizeof(T);
  static constexpr int NCH = RB / 16;
  static constexpr int LPR = NCH < 32 ? NCH : 32;
  static constexpr int EPW = 32 / LPR;
  static constexpr int CPL = NCH / LPR;
  // edges gathered per slot before they are consumed: keeps ~2 KB of K and
  // ~2 KB of V per warp in flight whatever the row size
  static constexpr int U0 = 4 / CPL > 0 ? 4 / CPL : 1;
  static constexpr int U = U0 * EPW <= 32 ? U0 : 32 / EPW;
  static constexpr int B = U * EPW;  // edges per sub-batch (divides 32)
  static_assert(RB % 16 == 0 && NCH >= 2, "row must hold at least two 16-byte chunks");
  static_assert(NCH <= 32 || NCH % 32 == 0, "rows above 512 B must be multiples of 512 B");
  static_assert(32 % B == 0, "sub-batch must divide 32");
};

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
// 16-byte chunk loads / stores with conversion to fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ldcg16(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

template <typename T>
struct Cvt;

template <>
struct Cvt<float> {
  static constexpr int VEC = 4;
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static uint4 from_f32(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct Cvt<__nv_bfloat16> {
  static constexpr int VEC = 8;
  __device__ __forceinline__ static void pair(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f) {
    pair(u.x, f[0], f[1]);
    pair(u.y, f[2], f[3]);
    pair(u.z, f[4], f[5]);
    pair(u.w, f[6], f[7]);
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&b);
  }
  __device__ __forceinline__ static uint4 from_f32(const float* f) {
    return make_uint4(pack(f[0], f[1]), pack(f[2], f[3]), pack(f[4], f[5]), pack(f[6], f[7]));
  }
};

// Sum over the LPH consecutive lanes of a head (LPH a power of two <= 32).
__device__ __forceinline__ float head_sum(float x, int lph) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
    if (o < lph) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

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
