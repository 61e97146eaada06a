// gdn_step_fused.cu -- instances of the fused verify step (conv + recurrence + persist).
#include "gdn_step_dispatch.cuh"

namespace lbx {

int launch_step_fused(const StepArgs &A, int d, cudaStream_t st) {
  switch (d) {
    case 32: return launch_step_d<32, true, true, false>(A, st);
    case 64: return launch_step_d<64, true, true, false>(A, st);
    case 128: return launch_step_d<128, true, true, false>(A, st);
  }
  return LBX_EINVAL;
}

}  // namespace lbx
