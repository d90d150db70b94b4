// attn_pipe.cuh -- thread layout and the per-warp asynchronous gather
// pipeline shared by the attention kernels.
//
// Thread layout.  A row (the H*D values of one node, RB bytes) is cut into
// TPR slices of PT = 32 bytes (64 for 2 KB rows); thread t of a group of TPR
// lanes owns slice t, i.e. NC consecutive 16-byte chunks.  A warp holds
// G = 32 / TPR groups and every group works on its OWN work item, so a warp
// advances G items at once (G = 4 for 256-byte rows).  A head whose D values
// fit in one slice needs no shuffle for its score; wider heads reduce over
// the lanes that share them.
//
// Degree binning.  The plan lists the work items (light nodes, heavy-node
// edge chunks) by decreasing edge count, so the G items of a bundle
// (consecutive items of that list) have (almost) equal length and their
// groups run in lockstep.
//
// Pipeline (one per warp, three levels, no inter-warp waits):
//   items  : the warp's next block of 32 / G bundles (one sorted item per
//            lane) is loaded into registers when the current block starts,
//            and stored to shared memory when it becomes current;
//   indices: stage t's descriptors (one per group: node, item, edge count,
//            FIRST/LAST flags) are generated and its source indices copied
//            (cp.async) 2S - 1 stages before t is computed;
//   rows   : stage t's rows (Q/K/V or their gradients' operands) are fetched
//            by the TMA engine S - 1 stages before t is computed, four rows
//            per tile::gather4 copy issued by one lane; completion is counted
//            in bytes on the stage slot's mbarrier.
// A stage holds SE edges of each of the G items.  Index copies complete
// through cp.async.wait_group (a hardware wait on the thread's own copies);
// the row barriers are polled with mbarrier.try_wait under an iteration
// limit, after which the kernel records an error instead of hanging.
#pragma once

#include "gattn_internal.cuh"
#include "tma.cuh"

namespace gattn {

constexpr int kStages = 2;           // row stages in flight + 1
constexpr int kRing = 2 * kStages;   // descriptor / index ring entries
constexpr int kUnit = 32;            // items per block of bundles
constexpr int kFirst = 1 << 29;
constexpr int kLast = 1 << 30;
constexpr int kCntMask = 0xffff;
constexpr int kSmemPerSm = 227 * 1024;

// SB: target bytes of gathered rows per stage (4 KB or 8 KB; the launcher
// picks by the plan's mean item length).
template <typename T, int RB, int SB>
struct Lay {
  static constexpr int RBYTES = RB;                 // bytes of a row
  static constexpr int VEC = 16 / (int)sizeof(T);  // elements per 16-byte chunk
  static constexpr int PT = RB <= 1024 ? 32 : RB / 32;
  static constexpr int NC = PT / 16;                // chunks per thread
  static constexpr int VP = NC * VEC / 2;           // float2 pairs per thread
  static constexpr int TPR = RB / PT;               // threads per row
  static constexpr int G = 32 / TPR;                // groups (items) per warp
  static constexpr int NCH = RB / 16;               // chunks per row
  // edges per item per stage: ~SB bytes of gathered rows per stage
  static constexpr int SE0 = SB / (2 * RB) / G;
  static constexpr int SE1 = SE0 < 1 ? 1 : SE0;
  static constexpr int SE2 = SE1 * G > 32 ? 32 / G : SE1;  // at most 32 edges per stage
  static constexpr int SE = SE2 * G < 4 ? 4 / G : SE2;     // whole 4-row gathers
  static constexpr int B = G * SE;                  // edges per stage
  static constexpr int QR = (G + 3) / 4 * 4;        // item-row indices per stage (whole 4-row sets)
  // Item rows held in a stage: whole 4-row gather sets when a warp holds 4
  // or more groups; one row per group otherwise, fetched by plain bulk
  // copies (no zero-filled pad rows taking shared memory).
  static constexpr bool IBULK = G < 4;
  static constexpr int IR = IBULK ? G : QR;
  // one gather moves 4 rows of BOXE elements; a row is NCOL such pieces
  static constexpr int HD = RB / (int)sizeof(T);
  static constexpr int BOXE = HD < kGatherBoxMax ? HD : kGatherBoxMax;
  static constexpr int NCOL = HD / BOXE;
  static constexpr int BOXB = BOXE * (int)sizeof(T);
  static constexpr int IDXB = (B * 4 + 15) / 16 * 16;
  // the warp's descriptor ring, index ring, item-row ring, unit buffer and
  // row barriers
  static constexpr int META =
      kRing * G * 16 + kRing * IDXB + kRing * QR * 4 + kUnit * 16 + 16 * ((kStages + 1) / 2);
  static_assert(TPR >= 1 && TPR <= 32 && 32 % TPR == 0, "thread layout");
  static_assert(B <= 32 && B % 4 == 0, "stage edges");
  // Byte offset of row byte x of row b in a region filled by 4-row gathers:
  // [b / 4][piece][b % 4][BOXB].
  __device__ __forceinline__ static int off(int b, int x) {
    if constexpr (NCOL == 1) return b * RB + x;
    else return (b / 4) * 4 * RB + (x / BOXB) * 4 * BOXB + (b % 4) * BOXB + x % BOXB;
  }
  // Byte offset of row byte x of item row b (the layout the item rows land in).
  __device__ __forceinline__ static int offI(int b, int x) {
    if constexpr (IBULK) return b * RB + x;
    else return off(b, x);
  }
  // Issue the gathers of rows r0..r3 into a region at row slot b0 (multiple of 4).
  __device__ __forceinline__ static void gather(uint8_t* region, int b0, const CUtensorMap* map,
                                                int r0, int r1, int r2, int r3, uint64_t* bar) {
#pragma unroll
    for (int pc = 0; pc < NCOL; ++pc)
      tma_gather4(region + b0 * RB + pc * 4 * BOXB, map, pc * BOXE, r0, r1, r2, r3, bar);
  }
  static constexpr int SET_BYTES = 4 * RB;  // bytes one 4-row gather set lands
  // per-node fp32 statistic rows (H <= RB/16 floats) are gathered 4 at a
  // time into SSB-byte sets (128-byte aligned), 4H bytes per row
  static constexpr int SSB = RB < 128 ? 128 : RB;
};

// Offsets are kept 128-byte aligned: tensor copies land on such addresses.
constexpr int align128(int x) { return (x + 127) / 128 * 128; }

// Warps per block: the count (1, 2, 4 or 8) that fits the most warps in an
// SM's shared memory (1 KB per block is reserved by the system); ties go to
// the larger block.
//
// Registers bound residency too: each of an SM's four sub-partitions holds
// 16,384 registers, allocated per warp in units of 256, so 16 resident warps
// need at most 128 registers a thread and 12 warps at most 168 (13 to 16
// warps need 4 per sub-partition, hence 128).  MINB asks the compiler for
// enough blocks per SM that registers never hold residency below what shared
// memory allows: 16 warps' worth when shared memory holds more than 12, 12
// when it holds 12, else the shared-memory count (the register cap follows
// from 65,536 / (MINB x block threads)).
template <int WARP_BYTES>
struct WarpsFor {
  static constexpr int fit(int w) { return (kSmemPerSm / (w * WARP_BYTES + 1024)) * w; }
  static constexpr int best(int w, int bw) { return w > 8 ? bw : best(2 * w, fit(w) >= fit(bw) ? w : bw); }
  static constexpr int value = best(1, 1);
  static constexpr int smem_warps = fit(value);
  static constexpr int target = smem_warps >= 16 ? 16 : (smem_warps >= 12 ? 12 : smem_warps);
  static constexpr int minb = target / value >= 1 ? target / value : 1;
};

// Blocks per SM a kernel asks the compiler for: the residency target above
// for the dot score.  GATv2 kernels need more registers: the 128- and
// 256-byte-row layouts with 8 KB stages take at most the 12-warp target
// (168 registers a thread, which they fit without spilling, as ptxas
// reports); the other GATv2 layouts spill under that cap and get none
// (8 resident warps at up to 255 registers).
template <int WARP_BYTES, int RB, int SB>
constexpr int min_blocks(int kind) {
  using W = WarpsFor<WARP_BYTES>;
  if (kind != GATTN_SCORE_GATV2) return W::minb;
  if (SB < 8192 || (RB != 128 && RB != 256)) return 1;
  return W::target > 12 ? (12 / W::value > 0 ? 12 / W::value : 1) : W::minb;
}

// ---------------------------------------------------------------------------
// async copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds16(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// mbarrier + TMA bulk copies (global -> this CTA's shared memory).  A wait
// suspends the warp in hardware for up to kSuspendNs per poll, so a waiting
// warp issues almost nothing; kWaitLimit polls bound a wait to about 0.2 s.
constexpr uint32_t kSuspendNs = 100000;
constexpr uint32_t kWaitLimit = 2000;
__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
// Bounded wait for the completion of the barrier phase with this parity
// (at most `limit` polls).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t limit = kWaitLimit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Item rows of a warp with fewer than 4 groups (Lay::IBULK): group b's row
// (index q[b], `pad` = none) is copied whole from `base` to region + b * RB.
template <typename L>
__device__ __forceinline__ int item_rows(int4 q, int pad) {
  const int r[4] = {q.x, q.y, q.z, q.w};
  int n = 0;
#pragma unroll
  for (int b = 0; b < L::G; ++b) n += r[b] != pad;
  return n;
}
template <typename L>
__device__ __forceinline__ void fetch_item_rows(uint8_t* region, const void* base, int4 q, int pad,
                                                uint64_t* bar) {
  const int r[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int b = 0; b < L::G; ++b)
    if (r[b] != pad)
      bulk_g2s(region + b * L::RBYTES, static_cast<const uint8_t*>(base) + int64_t(r[b]) * L::RBYTES,
               L::RBYTES, bar);
}

// ---------------------------------------------------------------------------
// 16-byte chunk <-> float2 pairs
// ---------------------------------------------------------------------------
template <typename T>
struct Pairs;

template <>
struct Pairs<__nv_bfloat16> {
  static constexpr int P = 4;  // pairs per chunk
  __device__ __forceinline__ static void load(const uint4& u, float2* f) {
    f[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
    f[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    f[2] = make_float2(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
    f[3] = make_float2(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
  }
  __device__ __forceinline__ static uint32_t pack(float2 v) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&b);
  }
  __device__ __forceinline__ static uint4 store(const float2* f) {
    return make_uint4(pack(f[0]), pack(f[1]), pack(f[2]), pack(f[3]));
  }
};

template <>
struct Pairs<float> {
  static constexpr int P = 2;
  __device__ __forceinline__ static void load(const uint4& u, float2* f) {
    f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
  __device__ __forceinline__ static uint4 store(const float2* f) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                      __float_as_uint(f[1].y));
  }
};

__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2s(float s) { return make_float2(s, s); }
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2abs(float2 a) { return make_float2(fabsf(a.x), fabsf(a.y)); }

// GATv2 LeakyReLU with slope s written as c1 z + c2 |z|, c1 = (1 + s) / 2,
// c2 = (1 - s) / 2 (exact at z = 0, no branch).  Its derivative, s + (1 - s)
// [z > 0], makes a gradient sum_j ds_j a LReLU'(z_j) equal to
// a (s sum_j ds_j + (1 - s) sum_{j: z_j > 0} ds_j): a kernel can accumulate
// the per-head sum of ds and the per-element sum over z > 0, and combine
// them once per work item.

// The heads a lane's NC chunks belong to: NC / CPH of them when a head is
// narrower than the lane's slice, else one (the lane holds part of a head).
// Per-head quantities (running max, sum, probabilities) are kept once per
// lane head, not once per chunk.
template <int NC, int CPH>
struct LaneHeads {
  static constexpr int N = CPH >= NC ? 1 : NC / CPH;  // heads per lane
  static constexpr int CPL = NC / N;                  // chunks per lane head
  __device__ __forceinline__ static constexpr int of(int c) { return c / CPL; }
};

// Per-lane-head totals y[LaneHeads::N] of per-lane-head float2 partial sums
// x2[LaneHeads::N] (the chunks of a lane head already accumulated into one
// pair, in chunk order): heads wider than a lane reduce over CPH / NC lanes.
// Every lane of the warp must call this (it may shuffle).  Every dot product
// of one kind (dO . v and dO . O in particular) goes through the same
// accumulation order, so equal inputs give bitwise equal sums.
template <int NC, int CPH>
__device__ __forceinline__ void head_sums2(const float2* x2, float* y) {
  using LH = LaneHeads<NC, CPH>;
#pragma unroll
  for (int j = 0; j < LH::N; ++j) y[j] = x2[j].x + x2[j].y;
  if constexpr (CPH > NC) {
#pragma unroll
    for (int o = 1; o < CPH / NC; o <<= 1) y[0] += __shfl_xor_sync(0xffffffffu, y[0], o);
  }
}

// ---------------------------------------------------------------------------
// the warp's cursor: bundles -> stages
// ---------------------------------------------------------------------------
// Bundle b is sorted items [b*G, b*G + G).  Bundles go to the W warps of the
// grid in rounds, in snake order (round r: bundles rW .. rW + W - 1, to warps
// 0..W-1 on even rounds and W-1..0 on odd ones).  With bundles sorted by
// decreasing length this is the classic longest-first greedy schedule: every
// warp ends up with nearly the same number of edges, deterministically and
// without atomics.  A warp's next 32/G bundles (one item per lane) are loaded
// into registers one such block ahead of use.
//
// Edge slots.  With RES = 0, edge k of group g sits in slot g * SE + k and
// the item rows of starting items have a region of their own.  With RES > 0
// ("inline" item rows), edge k of group g sits in slot k * G + g, so that
// edge k of every group forms whole 4-row gather sets (G >= 4), and the
// stage in which a bundle starts carries only SE - RES edges per group: its
// last RES edge positions hold the starting items' rows instead (the kernel
// gathers them there from the item tensors).  No stage then reserves shared
// memory for item rows that only the first stage of an item needs.
template <int G, int SE, int RES = 0>
struct BundleCursor {
  static constexpr int B = G * SE;
  static constexpr int R = kUnit / G;  // bundles per block
  static_assert(RES == 0 || (G >= 4 && SE > RES), "inline item rows need whole sets and an edge");
  __device__ __forceinline__ static constexpr int slot(int g, int k) {
    return RES > 0 ? k * G + g : g * SE + k;
  }
  const int4* sorted;     // items by decreasing length: (node, e0, e1, item index)
  const int32_t* idx;     // CSR sources (or CSC destinations)
  int pad;                // row index of unused gather slots (zero-filled)
  int64_t n_items, n_bundles, W, w, r_next;
  int4* s_items;          // [kUnit] current block of bundles, shared memory
  int4 pf;                // next block's item of this lane
  bool live;
  int bi, off, maxlen;

  __device__ __forceinline__ int64_t bundle_of(int64_t r) const {
    return r * W + ((r & 1) ? (W - 1 - w) : w);
  }
  __device__ __forceinline__ void prefetch(int lane) {
    const int64_t b = bundle_of(r_next + lane / G);
    const int64_t i = b * G + lane % G;
    pf = (b < n_bundles && i < n_items) ? sorted[i] : make_int4(-1, 0, 0, -1);
  }
  __device__ __forceinline__ void advance(int lane) {
    __syncwarp();
    live = bundle_of(r_next) < n_bundles;
    if (live) {
      s_items[lane] = pf;
      bi = 0;
      off = 0;
      r_next += R;
      prefetch(lane);
    }
    __syncwarp();
    if (live) maxlen = s_items[0].z - s_items[0].y;
  }
  __device__ __forceinline__ void start(const int4* sorted_, int64_t n_items_, const int32_t* idx_,
                                        int pad_, int64_t warp, int64_t nwarps, int4* s_items_,
                                        int lane) {
    sorted = sorted_;
    idx = idx_;
    pad = pad_;
    n_items = n_items_;
    n_bundles = (n_items_ + G - 1) / G;
    W = nwarps;
    w = warp;
    r_next = 0;
    s_items = s_items_;
    prefetch(lane);
    advance(lane);
  }

  // Generate the next stage into ring slot (desc[G], ix[B], qix[QR]): lane
  // g < G writes group g's descriptor {node (-1 idle, -3 end), item,
  // count|flags, first edge}; lane b < B copies the source index of slot b
  // (pad in unused slots); qix[g] is the node of an item that starts here,
  // else pad.  The issuing lane then reads whole 4-row sets from ix / qix.
  template <int QR>
  __device__ __forceinline__ void generate(int4* desc, int* ix, int* qix, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    int4 d = make_int4(-1, 0, 0, 0);
    if (!live) {
      if (lane < G) desc[lane] = make_int4(-3, 0, 0, 0);
      return;
    }
    const int step = off == 0 ? SE - RES : SE;  // edges per item in this stage
    if (lane < G) {
      const int4 it = s_items[bi + lane];
      const int len = it.z - it.y;
      if (it.x >= 0 && (off < len || (off == 0 && len == 0))) {
        const int cnt = min(step, len - off);
        const int fl = (off == 0 ? kFirst : 0) | (off + step >= len ? kLast : 0);
        d = make_int4(it.x, it.w, cnt | fl, it.y + off);
      }
      desc[lane] = d;
    }
    if (lane < QR) qix[lane] = (d.x >= 0 && (d.z & kFirst)) ? d.x : pad;
    const int g = RES > 0 ? lane % G : (lane / SE) & 31;
    const int k = RES > 0 ? lane / G : lane % SE;
    const int es = __shfl_sync(FULL, d.w, g);
    const int cn = __shfl_sync(FULL, d.x >= 0 ? (d.z & kCntMask) : 0, g);
    if (lane < B) {
      if (k < cn) cp_async4(ix + lane, idx + es + k);
      else ix[lane] = pad;
    }
    off += step;
    if (off >= maxlen) {
      bi += G;
      off = 0;
      // the rest of a block is empty once one of its bundles is
      if (bi >= kUnit || s_items[bi].x < 0) advance(lane);
      else maxlen = s_items[bi].z - s_items[bi].y;
    }
  }
};

// ---------------------------------------------------------------------------
// merge trees of heavy nodes
// ---------------------------------------------------------------------------
// Lanes of group g (TPR consecutive lanes) as a shuffle mask.
template <int TPR>
__device__ __forceinline__ unsigned group_mask(int g) {
  return TPR == 32 ? 0xffffffffu : (((1u << TPR) - 1u) << (g * TPR));
}

struct Tree {
  const int32_t* parent;  // [n_leaves + n_inner], -1 at a root
  const int2* kids;       // [n_inner]: (first child slot, count)
  int64_t n_leaves;       // slots [0, n_leaves) are the chunks
  int32_t* cnt;           // [n_inner] arrivals, zero between calls
};

// Climb the merge tree from leaf `slot` with the group's partial state.
// While the slot has a parent: store(slot) publishes the state, the group
// fences and counts its arrival at the parent; the group that arrives last
// loads the parent's children (merge(first, count), in slot order) into its
// state and continues from the parent.  Returns true for the one group that
// ends at the root holding the complete result.  Called by all lanes of a
// group and by no other lane; nothing waits.
template <class Merge, class Store>
__device__ __forceinline__ bool climb(const Tree& tr, int slot, unsigned gmask, int leader,
                                      bool is_leader, Merge merge, Store store) {
  for (;;) {
    const int par = tr.parent[slot];
    if (par < 0) return true;
    store(slot);
    __threadfence();
    __syncwarp(gmask);
    int old = 0;
    if (is_leader) old = atomicAdd(tr.cnt + (par - tr.n_leaves), 1);
    old = __shfl_sync(gmask, old, leader);
    const int2 kd = tr.kids[par - tr.n_leaves];
    if (old != kd.y - 1) return false;
    __threadfence();
    merge(kd.x, kd.y);
    __syncwarp(gmask);
    if (is_leader) tr.cnt[par - tr.n_leaves] = 0;
    slot = par;
  }
}

// Per-warp ring bookkeeping shared by the kernels' main loops.
template <typename L, int STAGE>
struct Ring {
  uint8_t* data;  // [kStages][STAGE]
  int4* desc;     // [kRing][G]
  uint8_t* ix;    // [kRing][IDXB]
  int* qix;       // [kRing][QR]
  int4* items;    // [kUnit]
  uint64_t* bar;  // [kStages] row barriers
  __device__ __forceinline__ void init(uint8_t* base, int lane) {
    data = base;
    desc = reinterpret_cast<int4*>(base + kStages * STAGE);
    ix = reinterpret_cast<uint8_t*>(desc + kRing * L::G);
    qix = reinterpret_cast<int*>(ix + kRing * L::IDXB);
    items = reinterpret_cast<int4*>(qix + kRing * L::QR);
    bar = reinterpret_cast<uint64_t*>(items + kUnit);
    if (lane == 0) {
      for (int k = 0; k < kStages; ++k) mbar_init(bar + k, 1);
      mbar_init_fence();
    }
    __syncwarp();
  }
  __device__ __forceinline__ void release(int lane) {
    __syncwarp();
    if (lane == 0)
      for (int k = 0; k < kStages; ++k) mbar_inval(bar + k);
    __syncwarp();
  }
  __device__ __forceinline__ uint64_t* bar_at(int t) { return bar + (t % kStages); }
  // Wait for stage t's rows, polling at most `limit` times.  On a failed
  // (timed-out) wait, record it in *err and wait again, bounded by the normal
  // limit, for the rows of every stage issued from t on (stage t itself
  // included), so that no copy into this warp's ring is still in flight when
  // the warp leaves; returns false.
  __device__ __forceinline__ bool wait_rows(int t, int32_t* err, int lane,
                                            uint32_t limit = kWaitLimit) {
    if (mbar_wait(bar_at(t), (t / kStages) & 1, limit)) return true;
    if (lane == 0) atomicOr(err, 1);
    for (int u = t; u < t + kStages; ++u)
      if (desc_at(u)[0].x != -3) mbar_wait(bar_at(u), (u / kStages) & 1);
    cp_async_wait<0>();
    return false;
  }
  // Poll limit of stage t's wait: a launch with `fail_first` set gives its
  // warps' first wait no polls at all (the failure path run on purpose).
  __device__ __forceinline__ static uint32_t limit_at(int t, int fail_first) {
    return (t == 0 && fail_first) ? 0u : kWaitLimit;
  }
  __device__ __forceinline__ int4* desc_at(int t) { return desc + (t % kRing) * L::G; }
  __device__ __forceinline__ int* ix_at(int t) {
    return reinterpret_cast<int*>(ix + (t % kRing) * L::IDXB);
  }
  __device__ __forceinline__ int* qix_at(int t) { return qix + (t % kRing) * L::QR; }
  // rows of 4-row set q4 of stage t's items / e4 of its edges
  __device__ __forceinline__ int4 qset(int t, int q4) {
    return reinterpret_cast<const int4*>(qix_at(t))[q4];
  }

  __device__ __forceinline__ int4 eset(int t, int e4) {
    return reinterpret_cast<const int4*>(ix_at(t))[e4];
  }
  // Generate stage t with the cursor.
  template <class Cursor>
  __device__ __forceinline__ void generate(Cursor& cur, int t, int lane) {
    cur.template generate<L::QR>(desc_at(t), ix_at(t), qix_at(t), lane);
  }
  __device__ __forceinline__ uint8_t* stage_at(int t) { return data + (t % kStages) * STAGE; }
};

}  // namespace gattn
