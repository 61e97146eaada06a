// gdn_aux.cu -- the unfused tree conv and the unfused persist kernels.
#include "gdn_launch.h"
#include "gdn_step.cuh"

namespace lbx {

// Grids of the conv and persist kernels aim at one wave of resident CTAs
// (4 per SM at 64 registers x 256 threads on 152 SMs; the conv kernel is
// held to 64 registers for it), so that the per-CTA batch check and window
// walk are paid once per CTA, not per block.
constexpr int kAuxTargetCtas = 4 * 152;

// One 8-channel group of one head block over the nodes s, s+S, s+2S, ...: the
// group's taps are loaded once, then each node is a single round trip for
// its window rows.  The G8 threads of a head block sit in an aligned run of
// one warp and step through the same nodes, so the L2 norm is a shuffle over
// that run; every thread runs the same trip count, so the shuffle is uniform.
template <int D, int KK>
__device__ __forceinline__ void conv_group(const ConvArgs &A, const int *win, int N, int C,
                                           const uint16_t *x_lb, const uint16_t *w_l,
                                           const float *cache_s, float *qkv_lb, bool act, int hb,
                                           int c0, int s, int S) {
  constexpr int G8 = D / 8;
  float wt[8][KK];
  if (act) {
    conv_taps<KK>(wt, w_l, c0);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int t = 0; t < KK; ++t) wt[e][t] = 0.f;
  }
  const bool norm = hb < 2 * A.Hk;
  const int trips = (N + S - 1) / S;
  for (int k = 0; k < trips; ++k) {
    const int i = s + k * S;
    const bool on = act && i < N;
    float v8[8];
    if (on) {
      const int *wi = win + i * LBX_MAX_CONV_WIDTH;
      // cache rows are a suffix of the window, so a deepest entry that is an
      // x row means every row is one: K bf16 loads, no fp32 halves, no
      // per-row select (same products in the same order as conv_rows)
      if (wi[KK - 1] >= 0) {
        uint4 xr[KK];
#pragma unroll
        for (int j = 0; j < KK; ++j) xr[j] = ldg_u4(x_lb + (size_t)wi[j] * C + c0);
#pragma unroll
        for (int e = 0; e < 8; ++e) v8[e] = 0.f;
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          float xv[8];
          unpack8(xr[j], xv);
#pragma unroll
          for (int e = 0; e < 8; ++e) v8[e] = fmaf(wt[e][KK - 1 - j], xv[e], v8[e]);
        }
      } else {
        conv_rows<KK>(v8, wt, wi, x_lb, C, cache_s, c0);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v8[e] = silu_fast(v8[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v8[e] = 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
    for (int o = G8 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float scale = norm ? rsqrtf(ss + A.l2_eps) : 1.f;
    if (on) {
      float *dst = qkv_lb + (size_t)i * C + c0;
      stg_f4(dst, make_float4(scale * v8[0], scale * v8[1], scale * v8[2], scale * v8[3]));
      stg_f4(dst + 4, make_float4(scale * v8[4], scale * v8[5], scale * v8[6], scale * v8[7]));
    }
  }
}

// One CTA per (layer, request, group of head blocks of D channels); the
// group size is ceil((2*Hk+Hv) / gridDim.y), at most kThreads/(D/8) so that
// each of the group's 8-channel slices has a thread.  Head blocks are laid out
// q heads | k heads | v heads, matching the channel order, so block hb covers
// channels [hb*D, (hb+1)*D); the first 2*Hk blocks are normalised.  Thread t
// takes slice t % (nb*D/8) over the nodes s, s+S, ... with s = t / (nb*D/8)
// and S = kThreads / (nb*D/8).
template <int D>
__global__ void __launch_bounds__(kThreads, 4) tree_conv_kernel(const ConvArgs A) {
  constexpr int G8 = D / 8;  // threads per head block and node
  __shared__ int win[LBX_MAX_TREE_NODES * LBX_MAX_CONV_WIDTH];
  __shared__ int par_s[LBX_MAX_TREE_NODES];
  __shared__ int flag;
  const int tid = threadIdx.x;
  const int N = A.N, K = A.K;
  const int nhb = 2 * A.Hk + A.Hv;
  const int bpc = (nhb + (int)gridDim.y - 1) / (int)gridDim.y;
  const int hb0 = (int)blockIdx.y * bpc;
  if (hb0 >= nhb || bpc * G8 > kThreads) return;  // uniform over the CTA
  const int lbi = blockIdx.x;
  const int l = lbi / A.Bq, bq = lbi % A.Bq;
  const int32_t *par_b = A.parent + (size_t)bq * N;
  // the parents are staged in one parallel load (made visible by the
  // barriers of the batch check) so that the window walk stays on chip
  if (tid < N) par_s[tid] = par_b[tid];
  {
    int code = validate_batch(A.parent, A.slot, nullptr, A.Bq, N, A.n_slots, false, false, false);
    code = block_any_error(code, &flag);
    if (code) {
      if (tid == 0 && A.status) *A.status = code;
      return;
    }
  }
  const int C = nhb * D;
  const uint16_t *x_lb = A.x + (size_t)lbi * N * C;
  const uint16_t *w_l = A.conv_w + (size_t)l * C * K;
  const float *cache_s = A.conv_cache + ((size_t)l * A.n_slots + A.slot[bq]) * (K - 1) * C;
  float *qkv_lb = A.qkv + (size_t)lbi * N * C;
  for (int i = tid; i < N; i += kThreads) {
    int m = i, past = 0;
    for (int j = 0; j < K; ++j) {
      if (m >= 0) {
        win[i * LBX_MAX_CONV_WIDTH + j] = m;
        m = par_s[m];
      } else {
        ++past;
        win[i * LBX_MAX_CONV_WIDTH + j] = -1 - (K - 1 - past);
      }
    }
  }
  __syncthreads();
  const int nb = nhb - hb0 < bpc ? nhb - hb0 : bpc;
  const int ngr = nb * G8;
  const int S = kThreads / ngr;
  const int s = tid / ngr, g = tid % ngr;
  const bool act = s < S;
  const int hb = hb0 + g / G8;
  const int c0 = hb * D + (g % G8) * 8;
  switch (K) {
    case 4: conv_group<D, 4>(A, win, N, C, x_lb, w_l, cache_s, qkv_lb, act, hb, c0, s, S); break;
    case 3: conv_group<D, 3>(A, win, N, C, x_lb, w_l, cache_s, qkv_lb, act, hb, c0, s, S); break;
    case 2: conv_group<D, 2>(A, win, N, C, x_lb, w_l, cache_s, qkv_lb, act, hb, c0, s, S); break;
    default: conv_group<D, 1>(A, win, N, C, x_lb, w_l, cache_s, qkv_lb, act, hb, c0, s, S); break;
  }
}

// Grid (chunks, L*Bq), chunks chosen for at most kAuxTargetCtas CTAs in all
// (at least one chunk per (layer, request)).
// Copies the accepted node's snapshot of every head into the request's state
// slot (four 16-byte loads in flight per thread) and rewrites its conv window.
template <int D>
__global__ void __launch_bounds__(kThreads) tree_persist_kernel(const PersistArgs A) {
  __shared__ int crow[LBX_MAX_CONV_WIDTH];
  __shared__ int par_s[LBX_MAX_TREE_NODES];
  __shared__ int flag;
  const int tid = threadIdx.x;
  const int N = A.N, K = A.K;
  const int lbi = blockIdx.y;
  const int l = lbi / A.Bq, bq = lbi % A.Bq;
  const int32_t *par_b = A.parent + (size_t)bq * N;
  // parents staged in one parallel load, visible after the check's barriers
  if (tid < N) par_s[tid] = par_b[tid];
  {
    int code = validate_batch(A.parent, A.slot, A.accepted, A.Bq, N, A.n_slots, false, true, true);
    code = block_any_error(code, &flag);
    if (code) {
      if (tid == 0 && A.status) *A.status = code;
      return;
    }
  }
  const int C = (2 * A.Hk + A.Hv) * D;
  const int s = A.slot[bq], acc = A.accepted[bq];
  const uint16_t *x_lb = A.x + (size_t)lbi * N * C;
  if (tid == 0) {
    int depth_acc = 0;
    for (int m = acc; m > 0; m = par_s[m]) ++depth_acc;
    for (int r = 0; r < K - 1; ++r) {
      const int dist = K - 2 - r;
      int w;
      if (dist <= depth_acc) {
        int m = acc;
        for (int t = 0; t < dist; ++t) m = par_s[m];
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
  const size_t stride = (size_t)gridDim.x * kThreads;
  size_t idx = (size_t)blockIdx.x * kThreads + tid;
  for (; idx + 3 * stride < total4; idx += 4 * stride) {
    const float4 v0 = __ldcs(src + idx), v1 = __ldcs(src + idx + stride),
                 v2 = __ldcs(src + idx + 2 * stride), v3 = __ldcs(src + idx + 3 * stride);
    __stcs(dst + idx, v0);
    __stcs(dst + idx + stride, v1);
    __stcs(dst + idx + 2 * stride, v2);
    __stcs(dst + idx + 3 * stride, v3);
  }
  for (; idx < total4; idx += stride) __stcs(dst + idx, __ldcs(src + idx));
  for (size_t c = (size_t)blockIdx.x * kThreads + tid; c < (size_t)C; c += stride)
    persist_conv_channel((int)c, K, C, crow, x_lb, cache, cache);
}

template <int D>
static int launch_conv_d(const ConvArgs &A, cudaStream_t st) {
  const int nhb = 2 * A.Hk + A.Hv, lbq = A.L * A.Bq;
  int groups = kAuxTargetCtas / lbq;
  if (groups < 1) groups = 1;
  if (groups > nhb) groups = nhb;
  // a power of two, so that the CTA's 8-channel slices (bpc * D/8) divide
  // its threads and none idles; at most one slice per thread
  const int want = (nhb + groups - 1) / groups;
  int bpc = 1;
  while (bpc < want && bpc * 2 <= kThreads / (D / 8)) bpc *= 2;
  dim3 grid(lbq, (nhb + bpc - 1) / bpc);
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
  const int lbq = A.L * A.Bq;
  unsigned chunks = (unsigned)(kAuxTargetCtas / lbq);
  if (chunks < 1u) chunks = 1u;
  if (chunks > gx) chunks = gx;
  if (chunks > 1024u) chunks = 1024u;
  dim3 grid(chunks, lbq);
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
