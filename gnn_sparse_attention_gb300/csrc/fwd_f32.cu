// fwd_f32.cu -- fwd kernels instantiated for float I/O (one translation
// unit per pass and dtype so the library compiles in parallel).
#include "attn_launch.cuh"

namespace gattn {

gattn_status launch_fwd_f32(int rb, int kind, const FwdParams& p, int num_sms, cudaStream_t st,
                                  int* grid_out) {
  return Launch<float>::fwd(rb, kind, p, num_sms, st, grid_out);
}

}  // namespace gattn
