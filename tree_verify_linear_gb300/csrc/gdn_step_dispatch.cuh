// gdn_step_dispatch.cuh -- picks the step-kernel instance for (d, node capacity).
//
// Row block R: 64 rows for d = 64 and 128 (two or one blocks per head), 32
// rows for d = 32.  The product tile has CG = 256 / (R/4) column groups and
// TC columns per thread, TC the smallest of {1,2,3,4,6,8} with CG*TC >= 2*cap.
#pragma once

#include "gdn_launch.h"
#include "gdn_step.cuh"

namespace lbx {

template <int D>
struct RowBlock {
  static constexpr int R = D >= 64 ? 64 : 32;
  static constexpr int CG = kThreads / (R / 4);
};

inline int pick_tc(int cg, int cap) {
  const int need = (2 * cap + cg - 1) / cg;
  const int opts[6] = {1, 2, 3, 4, 6, 8};
  for (int t : opts)
    if (t >= need) return t;
  return 0;
}

template <int D, int TC, bool F, bool P, bool S>
int launch_step_instance(const StepArgs &A, cudaStream_t st) {
  constexpr int R = RowBlock<D>::R;
  constexpr int CG = RowBlock<D>::CG;
  const StepLayout Ly = step_layout(D, R, TC, CG, A.cap);
  auto kern = gdn_step_kernel<D, R, TC, F, P, S>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly.total) !=
      cudaSuccess)
    return LBX_ECUDA;
  const long long grid = (long long)A.L * A.Bq * A.Hv * (D / R);
  if (grid <= 0 || grid > 0x7fffffffLL) return LBX_EINVAL;
  kern<<<(unsigned)grid, kThreads, Ly.total, st>>>(A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}

template <int D, bool F, bool P, bool S>
int launch_step_d(const StepArgs &A, cudaStream_t st) {
  switch (pick_tc(RowBlock<D>::CG, A.cap)) {
    case 1: return launch_step_instance<D, 1, F, P, S>(A, st);
    case 2: return launch_step_instance<D, 2, F, P, S>(A, st);
    case 3: return launch_step_instance<D, 3, F, P, S>(A, st);
    case 4: return launch_step_instance<D, 4, F, P, S>(A, st);
    case 6: return launch_step_instance<D, 6, F, P, S>(A, st);
    case 8: return launch_step_instance<D, 8, F, P, S>(A, st);
  }
  return LBX_EINVAL;
}

}  // namespace lbx
