// gdn_common.cuh -- small device helpers shared by the tree-verify kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lbx.h"

namespace lbx {

constexpr int kThreads = 256;

// bf16 bit pattern -> float (exact widening).
__device__ __forceinline__ float bf2f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

// The two bf16 values packed in one 32-bit word (low half first in memory).
__device__ __forceinline__ void bf2x2(uint32_t w, float &lo, float &hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&v)[8]) {
  bf2x2(u.x, v[0], v[1]);
  bf2x2(u.y, v[2], v[3]);
  bf2x2(u.z, v[4], v[5]);
  bf2x2(u.w, v[6], v[7]);
}

// Read-only 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_u4(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ float4 ldg_f4(const void *p) {
  uint4 u = ldg_u4(p);
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                     __uint_as_float(u.w));
}

// 16-byte asynchronous global -> shared copy (L2 only).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Streaming 16-byte global store (written once, not re-read by this kernel).
__device__ __forceinline__ void stg_f4(void *p, const float4 &v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// XOR swizzle of 16-byte chunks inside each 128-byte group of a row: chunk q
// of row r lives at chunk (q & ~7) | ((q ^ r) & 7).  Eight consecutive rows
// reading the same logical chunk then hit eight different bank groups.
__device__ __forceinline__ int swz(int q, int r) { return (q & ~7) | ((q ^ r) & 7); }

__device__ __forceinline__ float4 f4_scale(float s, const float4 &a) {
  return make_float4(s * a.x, s * a.y, s * a.z, s * a.w);
}
__device__ __forceinline__ void f4_fma(float4 &acc, float s, const float4 &a) {
  acc.x = fmaf(s, a.x, acc.x);
  acc.y = fmaf(s, a.y, acc.y);
  acc.z = fmaf(s, a.z, acc.z);
  acc.w = fmaf(s, a.w, acc.w);
}
__device__ __forceinline__ float dot4(const float4 &a, const float4 &b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float y) { return y / (1.0f + expf(-y)); }
// SiLU through the hardware exponential and a fast divide (a few ulp; the
// conv outputs it feeds are compared at ~1e-4 relative).
__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.0f + __expf(-y)); }

// Structural check of the whole batch, done by every CTA so that all CTAs
// reach the same verdict without talking to each other.  Returns 0 or an
// LBX_* code (per thread; combine with block_any_error).
//   chain:          every parent array must be the chain parent[i] == i-1
//   check_accepted: accepted[b] in [0, N)
//   check_distinct: no two requests name the same slot
// The checks are spread over the threads first, first + stride, ... (the
// whole block by default).
__device__ __forceinline__ int validate_batch(const int32_t *parent, const int32_t *slot,
                                              const int32_t *accepted, int Bq, int N,
                                              int n_slots, bool chain, bool check_accepted,
                                              bool check_distinct, int first = -1,
                                              int stride = 0) {
  if (first < 0) {
    first = threadIdx.x;
    stride = blockDim.x;
  }
  int bad = 0;
  for (int idx = first; idx < Bq * N; idx += stride) {
    int i = idx % N;
    int p = parent[idx];
    bool ok = chain ? (p == i - 1) : (i == 0 ? p == -1 : (p >= 0 && p < i));
    if (!ok) bad = LBX_ETREE;
  }
  for (int b = first; b < Bq; b += stride) {
    int s = slot[b];
    if (s < 0 || s >= n_slots) bad = LBX_EINVAL;
    if (check_accepted) {
      int a = accepted[b];
      if (a < 0 || a >= N) bad = LBX_EINVAL;
    }
    if (check_distinct)
      for (int b2 = 0; b2 < b; ++b2)
        if (slot[b2] == s) bad = LBX_EINVAL;
  }
  return bad;
}

// Block-wide "did any thread see an error": returns the error code seen by
// some thread (0 if none).  Uses one int of shared memory.
__device__ __forceinline__ int block_any_error(int code, int *flag_smem) {
  if (threadIdx.x == 0) *flag_smem = 0;
  __syncthreads();
  if (code) atomicExch(flag_smem, code);
  __syncthreads();
  int r = *flag_smem;
  __syncthreads();
  return r;
}

}  // namespace lbx
