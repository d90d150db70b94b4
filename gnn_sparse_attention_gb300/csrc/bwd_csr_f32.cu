// bwd_csr_f32.cu -- bwd_csr kernels instantiated for float I/O (one translation
// unit per pass and dtype so the library compiles in parallel).
#include "attn_launch.cuh"

namespace gattn {

gattn_status launch_bwd_csr_f32(int rb, int kind, const BwdParams& p, int num_sms, cudaStream_t st,
                                  int* grid_out) {
  return Launch<float>::bwd_csr(rb, kind, p, num_sms, st, grid_out);
}

}  // namespace gattn
