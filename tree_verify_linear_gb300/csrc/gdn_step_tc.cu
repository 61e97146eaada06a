// gdn_step_tc.cu -- host launch of the tensor-core fused step (d = 128, tree
// mode, N <= 24): tensor map of the state, persistent grid of one CTA per SM.
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace lbx {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool have_encode() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

int sm_count() {
  constexpr int kMaxDev = 256;
  static int cache[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

template <int NMAX>
int launch_tc(const StepArgs &A, cudaStream_t st) {
  if (!have_encode()) return LBX_ECUDA;
  const int nsm = sm_count();
  if (nsm <= 0) return LBX_ECUDA;
  // the state viewed as a 2-D array [L * n_slots * Hv * 128 rows][128 fp32]
  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)kTcD,
                              (cuuint64_t)A.L * A.n_slots * A.Hv * kTcD};
  const cuuint64_t gstride[1] = {(cuuint64_t)kTcD * sizeof(float)};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t estride[2] = {1, 1};
  if (g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(A.state_in), gdim,
               gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return LBX_ECUDA;
  TcArgs T;
  T.s = A;
  T.n_tiles = A.L * A.Bq * A.Hv;
  auto kern = gdn_step_tc_kernel<NMAX>;
  constexpr int smem = TcLayout<NMAX>::total;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return LBX_ECUDA;
  const int grid = T.n_tiles < nsm ? T.n_tiles : nsm;
  kern<<<grid, kTcThreads, smem, st>>>(map, T);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}

}  // namespace

bool step_tc_supported(int d, int N, int chain) {
  return d == kTcD && !chain && N >= 1 && N <= 24;
}

int launch_step_tc(const StepArgs &A, cudaStream_t st) {
  if ((long long)A.L * A.n_slots * A.Hv * kTcD > 0x7fffffffLL) return LBX_EINVAL;
  if (A.N <= 8) return launch_tc<8>(A, st);
  if (A.N <= 16) return launch_tc<16>(A, st);
  if (A.N <= 24) return launch_tc<24>(A, st);
  return LBX_EINVAL;
}

}  // namespace lbx
