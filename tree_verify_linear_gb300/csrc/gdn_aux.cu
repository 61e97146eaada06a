// gdn_aux.cu -- the unfused tree conv and the unfused persist kernels.
#include "gdn_launch.h"
#include "gdn_step.cuh"

namespace lbx {

// One CTA per (layer, request, head block of D channels).  Head blocks are
// laid out q heads | k heads | v heads, matching the channel order, so block
// hb covers channels [hb*D, (hb+1)*D); the first 2*Hk blocks are normalised.
template <int D>
__global__ void __launch_bounds__(kThreads) tree_conv_kernel(const ConvArgs A) {
  constexpr int G8 = D / 8;  // threads per node
  __shared__ int win[LBX_MAX_TREE_NODES * LBX_MAX_CONV_WIDTH];
  __shared__ int flag;
  const int tid = threadIdx.x;
  const int N = A.N, K = A.K;
  {
    int code = validate_batch(A.parent, A.slot, nullptr, A.Bq, N, A.n_slots, false, false, false);
    code = block_any_error(code, &flag);
    if (code) {
      if (tid == 0 && A.status) *A.status = code;
      return;
    }
  }
  const int lbi = blockIdx.x, hb = blockIdx.y;
  const int l = lbi / A.Bq, bq = lbi % A.Bq;
  const int C = (2 * A.Hk + A.Hv) * D;
  const size_t lb = (size_t)lbi;
  const int32_t *par_b = A.parent + (size_t)bq * N;
  const uint16_t *x_lb = A.x + lb * N * C;
  const uint16_t *w_l = A.conv_w + (size_t)l * C * K;
  const float *cache_s = A.conv_cache + ((size_t)l * A.n_slots + A.slot[bq]) * (K - 1) * C;
  for (int i = tid; i < N; i += kThreads) {
    int m = i, past = 0;
    for (int j = 0; j < K; ++j) {
      if (m >= 0) {
        win[i * LBX_MAX_CONV_WIDTH + j] = m;
        m = par_b[m];
      } else {
        ++past;
        win[i * LBX_MAX_CONV_WIDTH + j] = -1 - (K - 1 - past);
      }
    }
  }
  __syncthreads();
  const bool norm = hb < 2 * A.Hk;
  const int units = N * G8;
  for (int base = 0; base < units; base += kThreads) {
    const int u = base + tid;
    const bool act = u < units;
    const int i = act ? u / G8 : 0, li = u % G8;
    const int c0 = hb * D + li * 8;
    float v8[8];
    if (act) {
      conv8(v8, win + i * LBX_MAX_CONV_WIDTH, K, x_lb, C, w_l, cache_s, c0);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v8[e] = 0.f;
    }
    float scale = 1.f;
    if (norm) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
      for (int o = G8 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      scale = rsqrtf(ss + A.l2_eps);
    }
    if (act) {
      float *dst = A.qkv + (lb * N + i) * C + c0;
      stg_f4(dst, make_float4(scale * v8[0], scale * v8[1], scale * v8[2], scale * v8[3]));
      stg_f4(dst + 4, make_float4(scale * v8[4], scale * v8[5], scale * v8[6], scale * v8[7]));
    }
  }
}

// Grid (chunks, L*Bq).  Copies the accepted node's snapshot of every head
// into the request's state slot and rewrites its conv window.
template <int D>
__global__ void __launch_bounds__(kThreads) tree_persist_kernel(const PersistArgs A) {
  __shared__ int crow[LBX_MAX_CONV_WIDTH];
  __shared__ int flag;
  const int tid = threadIdx.x;
  const int N = A.N, K = A.K;
  {
    int code = validate_batch(A.parent, A.slot, A.accepted, A.Bq, N, A.n_slots, false, true, true);
    code = block_any_error(code, &flag);
    if (code) {
      if (tid == 0 && A.status) *A.status = code;
      return;
    }
  }
  const int lbi = blockIdx.y;
  const int l = lbi / A.Bq, bq = lbi % A.Bq;
  const int C = (2 * A.Hk + A.Hv) * D;
  const int s = A.slot[bq], acc = A.accepted[bq];
  const int32_t *par_b = A.parent + (size_t)bq * N;
  const uint16_t *x_lb = A.x + (size_t)lbi * N * C;
  if (tid == 0) {
    int depth_acc = 0;
    for (int m = acc; m > 0; m = par_b[m]) ++depth_acc;
    for (int r = 0; r < K - 1; ++r) {
      const int dist = K - 2 - r;
      int w;
      if (dist <= depth_acc) {
        int m = acc;
        for (int t = 0; t < dist; ++t) m = par_b[m];
        w = m;
      } else {
        w = -1 - (depth_acc + 1 + r);
      }
      crow[r] = w;
    }
  }
  __syncthreads();
  const size_t total4 = (size_t)A.Hv * D * D / 4;
  const float4 *src =
      reinterpret_cast<const float4 *>(A.node_states + ((size_t)lbi * N + acc) * A.Hv * D * D);
  float4 *dst = reinterpret_cast<float4 *>(A.state + ((size_t)l * A.n_slots + s) * A.Hv * D * D);
  float *cache = A.conv_cache + ((size_t)l * A.n_slots + s) * (K - 1) * C;
  for (size_t idx = (size_t)blockIdx.x * kThreads + tid; idx < total4 + C;
       idx += (size_t)gridDim.x * kThreads) {
    if (idx < total4) dst[idx] = src[idx];
    else persist_conv_channel((int)(idx - total4), K, C, crow, x_lb, cache, cache);
  }
}

template <int D>
static int launch_conv_d(const ConvArgs &A, cudaStream_t st) {
  dim3 grid(A.L * A.Bq, 2 * A.Hk + A.Hv);
  tree_conv_kernel<D><<<grid, kThreads, 0, st>>>(A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}

int launch_tree_conv(const ConvArgs &A, int d, cudaStream_t st) {
  switch (d) {
    case 32: return launch_conv_d<32>(A, st);
    case 64: return launch_conv_d<64>(A, st);
    case 128: return launch_conv_d<128>(A, st);
  }
  return LBX_EINVAL;
}

template <int D>
static int launch_persist_d(const PersistArgs &A, cudaStream_t st) {
  const size_t work = (size_t)A.Hv * D * D / 4 + (size_t)(2 * A.Hk + A.Hv) * D;
  const unsigned gx = (unsigned)((work + kThreads - 1) / kThreads);
  dim3 grid(gx < 1024 ? gx : 1024, A.L * A.Bq);
  tree_persist_kernel<D><<<grid, kThreads, 0, st>>>(A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}

int launch_tree_persist(const PersistArgs &A, int d, cudaStream_t st) {
  switch (d) {
    case 32: return launch_persist_d<32>(A, st);
    case 64: return launch_persist_d<64>(A, st);
    case 128: return launch_persist_d<128>(A, st);
  }
  return LBX_EINVAL;
}

}  // namespace lbx
