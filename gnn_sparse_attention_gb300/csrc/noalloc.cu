// noalloc.cu -- gattn_fwd_noalloc: the forward pass without a caller workspace.
//
// gattn_fwd needs device scratch for the partial results of heavy-node
// chunks, and the caller normally provides it (gattn_workspace_size +
// its own allocation).  Some callers cannot allocate device memory at the
// point where they run the layer: code that lives under an external memory
// pool or allocator that it does not own, or a plugin host that hands it
// only the input and output tensors.  For them this entry point takes its
// scratch from one fixed array compiled into the library, so the call itself
// allocates nothing.
//
// The array holds kNoAllocScratchBytes.  It exists on every device that loads
// the library for as long as the process lives, it is shared by every call,
// and it keeps whatever the last call left in it (nothing in it has to start
// at zero: each chunk writes its partial before any chunk reads it).  Calls
// whose kernels overlap on the GPU (several streams, or several host
// threads) race on it, so they must be ordered.
#include <cmath>
#include <mutex>

#include "attn_launch.cuh"
#include "tma.cuh"

namespace gattn {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_fwd_scratch[kNoAllocScratchBytes];

// The array's device address, cached per CUDA context: a device reset (or a
// context other than the one the address was looked up in) can place the
// module's globals at another address.
struct CtxAddr {
  void* ctx;
  void* addr;
};
std::mutex g_mu;
CtxAddr g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = int (*)(void**);  // cuCtxGetCurrent(CUcontext*)

// The driver's current context (nullptr when there is none or the query is
// unavailable), reached through the runtime's entry-point lookup so that the
// library needs no link-time dependency on the driver library.
void* current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// The device address of the scratch array in the current context.  The name
// g_fwd_scratch in host code is only a stand-in, so the address is looked up
// with cudaGetSymbolAddress (with the device current) the first time a
// context calls, and cached for that context.
gattn_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_error("gattn_fwd_noalloc: no usable current device (%s)", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  void* ctx = current_context();
  CtxAddr& c = g_scratch[dev];
  if (!c.addr || !ctx || c.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_error("gattn_fwd_noalloc: cudaGetSymbolAddress failed (%s)", cudaGetErrorString(e));
      return GATTN_ERR_CUDA;
    }
    // the lookup makes the device's primary context current if none was
    c.ctx = ctx ? ctx : current_context();
    c.addr = p;
  }
  *out = c.addr;
  return GATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

}  // namespace

}  // namespace gattn

using namespace gattn;

extern "C" gattn_status gattn_fwd_noalloc(const gattn_plan* plan, int32_t H, int32_t D,
                                          gattn_dtype dtype, const void* Q, const void* K,
                                          const void* V, const gattn_score* score, void* out,
                                          float* lse, gattn_stream_t stream) {
  if (!plan || !score) {
    set_error("gattn_fwd_noalloc: plan and score must be non-null");
    return GATTN_ERR_INVALID_ARG;
  }
  const Plan& p = plan->p;
  const int es = dtype == GATTN_F32 ? 4 : (dtype == GATTN_BF16 ? 2 : 0);
  if (es == 0 || H <= 0 || D <= 0) {
    set_error("gattn_fwd_noalloc: bad dtype or head layout");
    return GATTN_ERR_INVALID_ARG;
  }
  const int64_t db = int64_t(D) * es, rb = int64_t(H) * db;
  if (!pow2(H) || !pow2(D) || db < 16 || db > 512 || rb < 32 || rb > 2048) {
    set_error("gattn_fwd_noalloc: unsupported head layout H=%d D=%d", H, D);
    return GATTN_ERR_UNSUPPORTED;
  }
  FwdParams f{};
  if (score->kind == GATTN_SCORE_DOT) {
    const float scale = score->scale != 0.f ? score->scale : 1.f / sqrtf(float(D));
    f.qmul = scale * kLog2e;
  } else if (score->kind == GATTN_SCORE_GATV2) {
    if (!score->a || !aligned(score->a, 4)) {
      set_error("gattn_fwd_noalloc: GATv2 score needs a device pointer a[H*D] (4-byte aligned)");
      return GATTN_ERR_INVALID_ARG;
    }
    f.qmul = 1.f;
    f.slope = score->neg_slope;
  } else {
    set_error("gattn_fwd_noalloc: unknown score kind %d", score->kind);
    return GATTN_ERR_INVALID_ARG;
  }
  if (p.N == 0) return GATTN_OK;
  if (!Q || !K || !V || !out || !aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) ||
      !aligned(out, 16)) {
    set_error("gattn_fwd_noalloc: tensors must be non-null, 16-byte aligned device pointers");
    return GATTN_ERR_INVALID_ARG;
  }
  if (!lse || !aligned(lse, 4)) {
    set_error("gattn_fwd_noalloc: lse must be a non-null, 4-byte aligned device pointer");
    return GATTN_ERR_INVALID_ARG;
  }
  // scratch: one partial (acc[HD], m[H], l[H], padded to 4 floats) per tree slot
  const int64_t HD = int64_t(H) * D;
  const int pstride = int((HD + 2 * H + 3) / 4 * 4);
  const size_t need = size_t(p.n_chunks + p.n_inner) * pstride * sizeof(float);
  if (need > kNoAllocScratchBytes) {
    set_error("gattn_fwd_noalloc: this plan and head layout need %zu bytes of scratch, more "
              "than the fixed %zu; use gattn_fwd with a workspace",
              need, kNoAllocScratchBytes);
    return GATTN_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  gattn_status s = scratch_address(&scratch);
  if (s != GATTN_OK) return s;

  const bool bf = dtype == GATTN_BF16;
  if (!encode_rows_map(&f.mq, Q, es, bf, p.N, HD) || !encode_rows_map(&f.mk, K, es, bf, p.N, HD) ||
      !encode_rows_map(&f.mv, V, es, bf, p.N, HD))
    return GATTN_ERR_CUDA;
  f.items = p.items;
  f.sorted = p.sorted;
  f.n_items = p.n_chunks + p.n_light;
  f.n_chunks = p.n_chunks;
  f.N = p.N;
  f.indices = p.indices;
  f.Q = Q;
  f.K = K;
  f.V = V;
  f.out = out;
  f.lse = lse;
  f.a = score->a;
  f.H = H;
  f.D = D;
  f.part = static_cast<float*>(scratch);
  f.pstride = pstride;
  f.tree = Tree{p.parent, p.kids, p.n_chunks, p.cnt_fwd};
  f.err = p.err;
  f.fail_first_wait = p.fail_first_wait;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = launch_fwd(dtype, int(rb), int(db), score->kind, stage_bytes(p.M, f.n_items), f,
                      p.num_sms, st, nullptr)) !=
      GATTN_OK)
    return s;
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("gattn_fwd_noalloc: launch failed: %s", cudaGetErrorString(e));
    return GATTN_ERR_CUDA;
  }
  return GATTN_OK;
}
