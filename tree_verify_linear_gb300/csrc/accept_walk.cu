// accept_walk.cu -- verify argmax and greedy acceptance walk on the device.
//
// Lucebox hub README, "GPU draft top-K & verify-argmax (DFlash)": the
// target's per-node argmax over the vocabulary decides which draft tokens are
// accepted, and is taken on the device from the logits buffer so that no
// vocab x nodes copy reaches the host.  Greedy acceptance (the same README's
// serving notes: temperature 0 gives the highest acceptance) walks the draft
// tree from the root, at node u moving to the lowest-index child whose draft
// token equals the target's choice at u.
//
// One launch.  CTA (b, n, s) reduces slice s of logits row (b, n) to a
// (value, index) pair (NaN below every number, lowest index among equals) and
// stores it in the workspace; the last CTA of request b to arrive (arrival
// counter in the workspace, cleared again by that CTA) reduces the slices of
// every node, links each node to its lowest-index matching child, finds the
// accepted node by pointer jumping along those links (the reachable nodes
// form one path, so the deepest is the largest index), and writes the
// results.  The logits are read once, with 16-byte loads, four in flight
// per thread.
#include <stdint.h>

#include "gdn_common.cuh"
#include "lbx.h"

namespace lbx {
namespace {

constexpr int kAccThreads = 256;
constexpr int kAccTargetCtas = 1024;  // CTAs one call aims at (slices of the rows)
constexpr int kAccMinSlice = 2048;    // fewest logits per slice

// 1 if value a at index ia ranks above value b at index ib.
__device__ __forceinline__ bool ranks_above(float a, int ia, float b, int ib) {
  const bool na = isnan(a), nb = isnan(b);
  if (na || nb) return na && nb ? ia < ib : nb;
  return a > b || (a == b && ia < ib);
}

// Best (value, index) so far; index kNone = nothing seen yet.
constexpr int kNone = 0x7fffffff;
struct Best {
  float v;
  int i;
};
__device__ __forceinline__ void take(Best &x, float v, int i) {
  if (i != kNone && (x.i == kNone || ranks_above(v, i, x.v, x.i))) x.v = v, x.i = i;
}
// Four consecutive values from index i on, visited after every lower index
// of this thread: without NaN a strict > keeps the lowest index of a tie.
__device__ __forceinline__ void take4(Best &x, const float4 &f, int i) {
  if (f.x == f.x && f.y == f.y && f.z == f.z && f.w == f.w) {
    if (x.i == kNone || !(x.v == x.v) || f.x > x.v) x.v = f.x, x.i = i;  // a number beats NaN
    if (f.y > x.v) x.v = f.y, x.i = i + 1;
    if (f.z > x.v) x.v = f.z, x.i = i + 2;
    if (f.w > x.v) x.v = f.w, x.i = i + 3;
  } else {
    take(x, f.x, i);
    take(x, f.y, i + 1);
    take(x, f.z, i + 2);
    take(x, f.w, i + 3);
  }
}
__device__ __forceinline__ Best warp_best(Best x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, x.v, o);
    const int i = __shfl_xor_sync(0xffffffffu, x.i, o);
    take(x, v, i);
  }
  return x;
}

struct AccArgs {
  int Bq, N, V, S;
  const float *logits;
  const int32_t *draft, *parent;
  int32_t *argmax_out, *accepted_out, *next_out, *status;
  uint2 *part;          // [Bq][N][S] (value bits, index)
  unsigned int *count;  // [Bq] arrival counters
};

__global__ void __launch_bounds__(kAccThreads) accept_walk_kernel(const AccArgs A) {
  extern __shared__ int sh[];  // [N] choices, [N] links, then (S > 1) the slice results
  __shared__ float red_v[kAccThreads / 32];
  __shared__ int red_i[kAccThreads / 32];
  __shared__ int flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = A.S, N = A.N, V = A.V;
  const int s = blockIdx.x % S, row = blockIdx.x / S, b = row / N;

  // ---- this CTA's slice of the row ----
  {
    const int lo = (int)(((long long)V * s) / S), hi = (int)(((long long)V * (s + 1)) / S);
    const float *r = A.logits + (size_t)row * V;
    Best x = {0.f, kNone};
    // scalar head up to a 16-byte boundary, float4 body, scalar tail
    const int mis = (int)(((uintptr_t)(r + lo) >> 2) & 3u);
    int a0 = lo + (mis ? 4 - mis : 0);
    if (a0 > hi) a0 = hi;
    const int nv = (hi - a0) >> 2, a1 = a0 + 4 * nv;
    for (int v = lo + tid; v < a0; v += kAccThreads) take(x, r[v], v);
    const float4 *r4 = reinterpret_cast<const float4 *>(r + a0);
    // four 16-byte loads in flight per thread, visited in index order
    int q = tid;
    for (; q + 3 * kAccThreads < nv; q += 4 * kAccThreads) {
      const float4 f0 = __ldcs(r4 + q), f1 = __ldcs(r4 + q + kAccThreads),
                   f2 = __ldcs(r4 + q + 2 * kAccThreads), f3 = __ldcs(r4 + q + 3 * kAccThreads);
      take4(x, f0, a0 + 4 * q);
      take4(x, f1, a0 + 4 * (q + kAccThreads));
      take4(x, f2, a0 + 4 * (q + 2 * kAccThreads));
      take4(x, f3, a0 + 4 * (q + 3 * kAccThreads));
    }
    for (; q < nv; q += kAccThreads) take4(x, __ldcs(r4 + q), a0 + 4 * q);
    for (int v = a1 + tid; v < hi; v += kAccThreads) take(x, r[v], v);
    x = warp_best(x);
    if (lane == 0) red_v[warp] = x.v, red_i[warp] = x.i;
    __syncthreads();
    if (warp == 0) {
      Best y = {0.f, kNone};
      if (lane < kAccThreads / 32) y.v = red_v[lane], y.i = red_i[lane];
      y = warp_best(y);
      if (lane == 0) {
        A.part[(size_t)row * S + s] = make_uint2(__float_as_uint(y.v), (unsigned)y.i);
        __threadfence();
        flag = atomicAdd(A.count + b, 1u) == (unsigned)(N * S - 1);
      }
    }
    __syncthreads();
    if (!flag) return;
  }

  // ---- last CTA of request b: choices, links, walk ----
  __threadfence();
  int *choice = sh, *link = sh + N;
  const int32_t *par = A.parent + (size_t)b * N, *dr = A.draft + (size_t)b * N;
  int bad = 0;
  const uint2 *pp = A.part + (size_t)b * N * S;
  if (S == 1) {
    for (int n = tid; n < N; n += kAccThreads) choice[n] = (int)__ldcg(pp + n).y;
  } else {
    // the slices' results, one load per thread, staged after the two arrays
    int *stage = sh + 2 * N;
    for (int k = tid; k < N * S; k += kAccThreads) {
      const uint2 u = __ldcg(pp + k);
      stage[2 * k] = (int)u.x;
      stage[2 * k + 1] = (int)u.y;
    }
    __syncthreads();
    for (int n = tid; n < N; n += kAccThreads) {
      Best y = {0.f, kNone};
      for (int k = 0; k < S; ++k)
        take(y, __int_as_float(stage[2 * (n * S + k)]), stage[2 * (n * S + k) + 1]);
      choice[n] = y.i;
    }
  }
  __syncthreads();
  for (int n = tid; n < N; n += kAccThreads) {
    const int p = par[n];
    if (n == 0 ? p != -1 : !(p >= 0 && p < n)) bad = 1;
    link[n] = 0x7fffffff;
  }
  bad = __syncthreads_or(bad);
  if (tid == 0) A.count[b] = 0u;  // every CTA of the request has arrived
  if (bad) {
    if (tid == 0 && A.status) *A.status = LBX_ETREE;
    return;
  }
  // link[u] = the lowest-index child of u that carries the choice at u
  for (int c = 1 + tid; c < N; c += kAccThreads)
    if (dr[c] == choice[par[c]]) atomicMin(link + par[c], c);
  __syncthreads();
  // up[c] = the parent of c if the walk steps from it to c, else -1 (the
  // root: 0), replacing the links; then pointer jumping: after ceil(log2 N)
  // rounds up[c] == 0 exactly for the nodes on the walk
  constexpr int kPer = (LBX_ACCEPT_MAX_NODES + kAccThreads - 1) / kAccThreads;
  int nu[kPer];
  {
    int k = 0;
    for (int c = tid; c < N; c += kAccThreads, ++k)
      nu[k] = c == 0 ? 0 : (link[par[c]] == c ? par[c] : -1);
    __syncthreads();
    k = 0;
    for (int c = tid; c < N; c += kAccThreads, ++k) link[c] = nu[k];
    __syncthreads();
  }
  for (int span = 1; span < N; span <<= 1) {
    int k = 0;
    for (int c = tid; c < N; c += kAccThreads, ++k) {
      const int u = link[c];
      nu[k] = u > 0 ? link[u] : u;
    }
    __syncthreads();
    k = 0;
    for (int c = tid; c < N; c += kAccThreads, ++k) link[c] = nu[k];
    __syncthreads();
  }
  int deepest = 0;
  for (int c = tid; c < N; c += kAccThreads)
    if (link[c] == 0 && c > deepest) deepest = c;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) deepest = max(deepest, __shfl_xor_sync(0xffffffffu, deepest, o));
  if (lane == 0) red_i[warp] = deepest;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < kAccThreads / 32; ++w) acc = max(acc, red_i[w]);
    A.accepted_out[b] = acc;
    A.next_out[b] = choice[acc];
  }
  if (A.argmax_out)
    for (int n = tid; n < N; n += kAccThreads) A.argmax_out[(size_t)b * N + n] = choice[n];
}

int slices(int Bq, int N, int V) {
  long long s = (kAccTargetCtas + (long long)Bq * N - 1) / ((long long)Bq * N);
  const long long smax = (V + kAccMinSlice - 1) / kAccMinSlice;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  return (int)s;
}

}  // namespace
}  // namespace lbx

extern "C" size_t lbx_accept_workspace_size(int Bq, int N, int V) {
  if (Bq < 1 || N < 1 || N > LBX_ACCEPT_MAX_NODES || V < 1) return 0;
  const size_t part = (size_t)Bq * N * lbx::slices(Bq, N, V) * sizeof(uint2);
  return ((part + 255) & ~(size_t)255) + (((size_t)Bq * 4 + 255) & ~(size_t)255);
}

extern "C" int lbx_accept_walk(int Bq, int N, int V, const float *logits, const int32_t *draft,
                               const int32_t *parent, int32_t *argmax_out,
                               int32_t *accepted_out, int32_t *next_out, void *workspace,
                               size_t workspace_bytes, int32_t *d_status, cudaStream_t stream) {
  const size_t need = lbx_accept_workspace_size(Bq, N, V);
  if (need == 0) return LBX_EINVAL;
  if ((long long)Bq * N * V > (1LL << 40)) return LBX_EINVAL;
  auto al = [](const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; };
  if (!logits || !al(logits, 4) || !draft || !al(draft, 4) || !parent || !al(parent, 4) ||
      !accepted_out || !al(accepted_out, 4) || !next_out || !al(next_out, 4) ||
      (argmax_out && !al(argmax_out, 4)) || (d_status && !al(d_status, 4)) || !workspace ||
      !al(workspace, 16) || workspace_bytes < need)
    return LBX_EINVAL;
  lbx::AccArgs A;
  A.Bq = Bq, A.N = N, A.V = V, A.S = lbx::slices(Bq, N, V);
  A.logits = logits, A.draft = draft, A.parent = parent;
  A.argmax_out = argmax_out, A.accepted_out = accepted_out, A.next_out = next_out;
  A.status = d_status;
  A.part = static_cast<uint2 *>(workspace);
  const size_t part = (size_t)Bq * N * A.S * sizeof(uint2);
  A.count = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(workspace) +
                                             ((part + 255) & ~(size_t)255));
  const long long grid = (long long)Bq * N * A.S;
  if (grid > 0x7fffffffLL) return LBX_EINVAL;
  const size_t smem = ((size_t)2 * N + (A.S > 1 ? (size_t)2 * N * A.S : 0)) * sizeof(int);
  if (smem > 48 * 1024) return LBX_EINVAL;  // not reached: S > 1 only while Bq N < 1024
  lbx::accept_walk_kernel<<<(unsigned)grid, lbx::kAccThreads, smem, stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}
