// gdn_step_tc.cu -- host launch of the tensor-core fused step (d = 128, tree
// mode, N <= 24): tensor maps of the state, the raw inputs and the conv cache;
// the prep kernel (one CTA per key head), then the step kernel on a
// persistent grid of two CTAs per SM.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gdn_launch.h"
#include "gdn_tc.cuh"
#include "gdn_tc_prep.cuh"
#include "gdn_chain_tc.cuh"

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

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, int esize, const void *base,
               uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swz) {
  const cuuint64_t gdim[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)inner * esize};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return g_encode(map, dt, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMAX>
int launch_tc(const StepArgs &A, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (ws == nullptr || ws_bytes < tc_workspace_bytes<NMAX>(A.L, A.Bq, A.Hk, A.Hv)) return LBX_EINVAL;
  if (((uintptr_t)ws & 15u) != 0) return LBX_EINVAL;
  if (!have_encode()) return LBX_ECUDA;
  const int nsm = sm_count();
  if (nsm <= 0) return LBX_ECUDA;
  const int C = (2 * A.Hk + A.Hv) * kTcD;
  TcMaps maps;
  std::memset(&maps, 0, sizeof maps);
  // the state as [L * n_slots * Hv * 128 rows][128 fp32], 32-column boxes
  if (!encode_2d(&maps.state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A.state_in, kTcD,
                 (uint64_t)A.L * A.n_slots * A.Hv * kTcD, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return LBX_ECUDA;
  // x as [L * Bq * N rows][C bf16]: one box = one 128-channel block of all nodes
  if (!encode_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, A.x, C, (uint64_t)A.L * A.Bq * A.N,
                 kTcD, A.N, CU_TENSOR_MAP_SWIZZLE_NONE))
    return LBX_ECUDA;
  // the conv cache as [L * n_slots * (K-1) rows][C fp32]: one box = the K-1
  // cached rows of a 128-channel block
  if (A.K > 1 && !encode_2d(&maps.cache, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A.conv_cache, C,
                            (uint64_t)A.L * A.n_slots * (A.K - 1), kTcD, A.K - 1,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
    return LBX_ECUDA;
  TcArgs T;
  T.s = A;
  T.n_tiles = A.L * A.Bq * A.Hv;
  T.ws = static_cast<unsigned char *>(ws);
  {
    auto prep = gdn_qk_prep_kernel<NMAX>;
    constexpr int psmem = PrepLayout<NMAX>::total;
    if (cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem) !=
        cudaSuccess)
      return LBX_ECUDA;
    prep<<<A.L * A.Bq * A.Hk, TcRes<NMAX>::prep_threads, psmem, st>>>(maps, T);
    if (cudaGetLastError() != cudaSuccess) return LBX_ECUDA;
  }
  auto kern = gdn_step_tc_kernel<NMAX>;
  constexpr int smem = TcLayout<NMAX>::smem_bytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return LBX_ECUDA;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return LBX_ECUDA;
  const int slots = TcRes<NMAX>::ctas * nsm;
  const int grid = T.n_tiles < slots ? T.n_tiles : slots;
  // programmatic stream serialization: the step kernel may start while the
  // prep kernel's last CTAs run, and waits for it before reading the workspace
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(TcRes<NMAX>::threads);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, kern, maps, T) != cudaSuccess) return LBX_ECUDA;
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}

int launch_chain(const StepArgs &A, cudaStream_t st) {
  if (!have_encode()) return LBX_ECUDA;
  const int nsm = sm_count();
  if (nsm <= 0) return LBX_ECUDA;
  const int C = (2 * A.Hk + A.Hv) * kTcD;
  ChainMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (!encode_2d(&maps.state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A.state_in, kTcD,
                 (uint64_t)A.L * A.n_slots * A.Hv * kTcD, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return LBX_ECUDA;
  // x as [L * Bq * N rows][C bf16]: one box = one 128-channel block of a
  // chunk's tokens and the 3 before it
  if (!encode_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, A.x, C, (uint64_t)A.L * A.Bq * A.N,
                 kTcD, kChainRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return LBX_ECUDA;
  if (A.K > 1 && !encode_2d(&maps.cache, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A.conv_cache, C,
                            (uint64_t)A.L * A.n_slots * (A.K - 1), kTcD, A.K - 1,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
    return LBX_ECUDA;
  ChainArgs T;
  T.s = A;
  T.n_seq = A.L * A.Bq * A.Hv;
  constexpr int smem = ChainLayout::total;
  if (cudaFuncSetAttribute(gdn_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return LBX_ECUDA;
  if (cudaFuncSetAttribute(gdn_chain_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return LBX_ECUDA;
  const int slots = kTcCtasPerSm * nsm;
  const int grid = T.n_seq < slots ? T.n_seq : slots;
  gdn_chain_tc_kernel<<<grid, kTcThreads, smem, st>>>(maps, T);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}

}  // namespace

bool chain_tc_supported(int d) { return d == kTcD; }

int launch_chain_tc(const StepArgs &A, cudaStream_t st) {
  if ((long long)A.L * A.n_slots * A.Hv * kTcD > 0x7fffffffLL) return LBX_EINVAL;
  if ((long long)A.L * A.Bq * A.N > 0x7fffffffLL) return LBX_EINVAL;
  return launch_chain(A, st);
}

bool step_tc_supported(int d, int N, int chain) {
  return d == kTcD && !chain && N >= 1 && N <= 64;
}

size_t step_tc_workspace_bytes(int L, int Bq, int Hk, int Hv, int N) {
  if (N <= 8) return tc_workspace_bytes<8>(L, Bq, Hk, Hv);
  if (N <= 16) return tc_workspace_bytes<16>(L, Bq, Hk, Hv);
  if (N <= 24) return tc_workspace_bytes<24>(L, Bq, Hk, Hv);
  if (N <= 32) return tc_workspace_bytes<32>(L, Bq, Hk, Hv);
  if (N <= 64) return tc_workspace_bytes<64>(L, Bq, Hk, Hv);
  return 0;
}

int launch_step_tc(const StepArgs &A, void *ws, size_t ws_bytes, cudaStream_t st) {
  if ((long long)A.L * A.n_slots * A.Hv * kTcD > 0x7fffffffLL) return LBX_EINVAL;
  if ((long long)A.L * A.Bq * A.N > 0x7fffffffLL) return LBX_EINVAL;
  if (A.N <= 8) return launch_tc<8>(A, ws, ws_bytes, st);
  if (A.N <= 16) return launch_tc<16>(A, ws, ws_bytes, st);
  if (A.N <= 24) return launch_tc<24>(A, ws, ws_bytes, st);
  if (A.N <= 32) return launch_tc<32>(A, ws, ws_bytes, st);
  if (A.N <= 64) return launch_tc<64>(A, ws, ws_bytes, st);
  return LBX_EINVAL;
}

}  // namespace lbx
