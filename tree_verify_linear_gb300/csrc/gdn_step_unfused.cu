// gdn_step_unfused.cu -- instances of the recurrence-only step (from a conv output),
// with and without per-node state snapshots.
#include "gdn_step_dispatch.cuh"

namespace lbx {

int launch_step_unfused(const StepArgs &A, int d, cudaStream_t st) {
  const bool snap = A.node_states != nullptr;
  switch (d) {
    case 32:
      return snap ? launch_step_d<32, false, false, true>(A, st)
                  : launch_step_d<32, false, false, false>(A, st);
    case 64:
      return snap ? launch_step_d<64, false, false, true>(A, st)
                  : launch_step_d<64, false, false, false>(A, st);
    case 128:
      return snap ? launch_step_d<128, false, false, true>(A, st)
                  : launch_step_d<128, false, false, false>(A, st);
  }
  return LBX_EINVAL;
}

int step_smem_bytes(int d, int cap) {
  switch (d) {
    case 32: {
      const int tc = pick_tc(RowBlock<32>::CG, cap);
      return tc ? step_layout(32, RowBlock<32>::R, tc, RowBlock<32>::CG, cap).total : 0;
    }
    case 64: {
      const int tc = pick_tc(RowBlock<64>::CG, cap);
      return tc ? step_layout(64, RowBlock<64>::R, tc, RowBlock<64>::CG, cap).total : 0;
    }
    case 128: {
      const int tc = pick_tc(RowBlock<128>::CG, cap);
      return tc ? step_layout(128, RowBlock<128>::R, tc, RowBlock<128>::CG, cap).total : 0;
    }
  }
  return 0;
}

}  // namespace lbx
