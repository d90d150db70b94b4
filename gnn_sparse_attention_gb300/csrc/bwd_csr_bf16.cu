// bwd_csr_bf16.cu -- bwd_csr kernels instantiated for __nv_bfloat16 I/O (one translation
// unit per pass and dtype so the library compiles in parallel).
#include "attn_launch.cuh"

namespace gattn {

gattn_status launch_bwd_csr_bf16(int rb, int kind, const BwdParams& p, int num_sms, cudaStream_t st,
                                  int* grid_out) {
  return Launch<__nv_bfloat16>::bwd_csr(rb, kind, p, num_sms, st, grid_out);
}

}  // namespace gattn
