// gdn_tc_prep.cuh -- per-key-head preparation for the tensor-core step.
//
// One CTA per (layer l, request b, key head): the q and k conv + SiLU + L2
// normalisation along each node's ancestor path (q scaled), written as the
// bf16 hi / lo [K|Q] operand image of the step kernel; the Gram entries
// k_j.k_n and k_j.q_n of every (node n, strict ancestor j) pair and k_n.q_n
// (from the same hi + lo values the tensor cores see); the new conv window of
// the key head's q and k channels, persisted in place (this CTA is the only
// reader and writer of those channels); and, by the CTAs of layer 0 and key
// head 0, the request's tree tables.  Everything lands in the caller's
// workspace and is bulk-copied by the step kernel, so the step kernel's tiles
// carry no per-key-head prologue and need no arrival counters.
#pragma once

#include "gdn_tc.cuh"

namespace lbx {

constexpr int kPrepThreads = 256;

// Tree tables of one request in the new labels (the accepted path, root
// first, takes labels 0..P-1; the other nodes follow in input order, so
// parents still precede children).  All NT threads of the CTA take part;
// named barrier 1 separates the steps.  porig: int [NMAX] scratch.
template <int NMAX, int NT>
__device__ void build_tables(int tid, int N, int K, int acc, const int32_t *par_b,
                             unsigned char *tb, int *porig) {
  using TL = TabLayout<NMAX>;
  unsigned char *pj = tb + TL::pj, *pn = tb + TL::pn, *ln = tb + TL::ln;
  int *par = reinterpret_cast<int *>(tb + TL::par);
  int *dep = reinterpret_cast<int *>(tb + TL::dep);
  int *off = reinterpret_cast<int *>(tb + TL::off);
  int *off2 = reinterpret_cast<int *>(tb + TL::off2);
  int *win = reinterpret_cast<int *>(tb + TL::win);
  int *n2o = reinterpret_cast<int *>(tb + TL::n2o);
  int *o2n = reinterpret_cast<int *>(tb + TL::o2n);
  int *crow = reinterpret_cast<int *>(tb + TL::crow);
  int *meta = reinterpret_cast<int *>(tb + TL::meta);
  if (tid < NMAX) {
    porig[tid] = tid < N ? par_b[tid] : -1;
    o2n[tid] = -1;
    n2o[tid] = 0;
  }
  ptx::named_sync(1, NT);
  if (tid == 0) {
    int P = 0;
    for (int m = acc; m >= 0; m = porig[m]) ++P;
    int p = P;
    for (int m = acc; m >= 0; m = porig[m]) {
      --p;
      n2o[p] = m;
      o2n[m] = p;
    }
    int c = P;
    for (int i = 0; i < N; ++i)
      if (o2n[i] < 0) {
        n2o[c] = i;
        o2n[i] = c;
        ++c;
      }
    meta[0] = P;
  }
  if (tid == 32) {
    for (int rr = 0; rr < 4; ++rr) crow[rr] = 0;
    window_sources(crow, K, acc, porig);
  }
  ptx::named_sync(1, NT);
  if (tid < NMAX) {
    // parent, depth and conv window rows in the new labels; taps j >= K
    // and padding nodes point at input row 0
    const int o = tid < N ? n2o[tid] : 0;
    par[tid] = tid < N && porig[o] >= 0 ? o2n[porig[o]] : -1;
    int d = 0;
    if (tid < N)
      for (int m = porig[o]; m >= 0; m = porig[m]) ++d;
    dep[tid] = d;
    int m = tid < N ? o : -2, past = 0;
    for (int j = 0; j < 4; ++j) {
      int w = 0;
      if (tid < N && j < K) {
        if (m >= 0) {
          w = m;
          m = porig[m];
        } else {
          ++past;
          w = -1 - (K - 1 - past);
        }
      }
      win[tid * 4 + j] = w;
    }
  }
  ptx::named_sync(1, NT);
  if (tid <= NMAX) {
    int o1 = 0, o2 = 0;
    for (int i = 0; i < N && i < tid; ++i) {
      o1 += dep[i];
      o2 += dep[i] + 1;
    }
    off[tid] = o1;
    off2[tid] = o2;
  }
  ptx::named_sync(1, NT);
  for (int i = tid; i < N; i += NT) {
    int j = par[i];
    for (int e = off[i]; e < off[i + 1]; ++e) {
      pj[e] = (unsigned char)j;
      pn[e] = (unsigned char)i;
      j = par[j];
    }
    for (int q = off2[i]; q < off2[i + 1]; ++q) ln[q] = (unsigned char)i;
  }
  if (tid == 0) {
    meta[1] = off2[N];
    meta[2] = off[N];
    meta[3] = 0;
  }
  ptx::named_sync(1, NT);
}

template <int NMAX>
__global__ void __launch_bounds__(kPrepThreads, 1)
    gdn_qk_prep_kernel(const __grid_constant__ TcMaps maps, const TcArgs T) {
  using Ly = TcLayout<NMAX>;
  using PL = PrepLayout<NMAX>;
  using CS = ConvStage<NMAX>;
  using TL = TabLayout<NMAX>;
  using GL = GramLayout<NMAX>;
  constexpr int NT = kPrepThreads, NC = Ly::NC, R1 = Ly::R1;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *B1 = smem + PL::b1;
  float *kqf = reinterpret_cast<float *>(smem + PL::kqf);
  unsigned char *sq = smem + PL::sq, *sk = smem + PL::sk;
  float *gkk = reinterpret_cast<float *>(smem + PL::gr + GL::gkk);
  float *gkq = reinterpret_cast<float *>(smem + PL::gr + GL::gkq);
  float *kqn = reinterpret_cast<float *>(smem + PL::gr + GL::kqn);
  unsigned char *tb = smem + PL::tb;
  int *porig = reinterpret_cast<int *>(smem + PL::porig);
  int *misc = reinterpret_cast<int *>(smem + PL::misc);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + PL::bar);
  const int tid = threadIdx.x;
  const int N = A.N, K = A.K, Hk = A.Hk, Hv = A.Hv, Bq = A.Bq;
  const int C = (2 * Hk + Hv) * kTcD;
  const uint32_t stg_bytes =
      (uint32_t)N * kTcD * 2 + (uint32_t)(K - 1) * kTcD * 4 + (uint32_t)kTcD * K * 2;

  // an invalid batch is reported by the step kernel; nothing is done here
  {
    const int code =
        validate_batch(A.parent, A.slot, A.accepted, Bq, N, A.n_slots, false, true, true);
    if (block_any_error(code, misc)) return;
  }
  const int g = blockIdx.x;
  const int kh = g % Hk, lbi = g / Hk;
  const int bq = lbi % Bq, l = lbi / Bq;
  const int slot_b = A.slot[bq];
  const int crow0 = (l * A.n_slots + slot_b) * (K - 1);

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(bar, 2 * stg_bytes);
    for (int which = 0; which < 2; ++which) {
      unsigned char *dst = which == 0 ? sq : sk;
      const int ch0 = (which * Hk + kh) * kTcD;
      ptx::tma_load_2d(dst + CS::x, &maps.x, ch0, lbi * N, bar);
      if (K > 1) ptx::tma_load_2d(dst + CS::c, &maps.cache, ch0, crow0, bar);
      ptx::bulk_load(dst + CS::w, A.conv_w + (size_t)l * C * K + (size_t)ch0 * K,
                     (uint32_t)kTcD * K * 2, bar);
    }
  }
  __syncthreads();
  build_tables<NMAX, NT>(tid, N, K, A.accepted[bq], A.parent + (size_t)bq * N, tb, porig);
  const int *win = reinterpret_cast<const int *>(tb + TL::win);
  const int *crow = reinterpret_cast<const int *>(tb + TL::crow);
  const unsigned char *pj = tb + TL::pj, *pn = tb + TL::pn;
  const int npair = reinterpret_cast<const int *>(tb + TL::meta)[2];
  if (!ptx::mbar_wait(bar, 0)) {
    if (A.status) *A.status = LBX_ETIMEOUT;
    (void)ptx::mbar_wait(bar, 0);  // the copies must land before the CTA exits
    return;
  }

  // q, then k: conv + SiLU + L2 norm -> operand rows (hi, lo) and fp32 hi + lo
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const unsigned char *cs = which == 0 ? sq : sk;
    constexpr int GQ = kTcD / 8;  // 16 threads per node, the same 8 channels for every node
    constexpr int U = (NMAX * GQ + NT - 1) / NT;
    static_assert(NT % GQ == 0, "channel group fixed per thread");
    const int li = tid % GQ;
    float wsl[8][LBX_MAX_CONV_WIDTH];
    conv_weights8<NMAX>(wsl, K, cs, li * 8);
#pragma unroll
    for (int p = 0; p < U; ++p) {
      const int u = p * NT + tid;
      const bool act = u < N * GQ;
      const int i = act ? u / GQ : 0;
      float v8[8];
      conv8_staged<NMAX>(v8, win + i * 4, wsl, cs, li * 8);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
      for (int o = GQ / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (act) {
        const float scale = rsqrtf(ss + A.l2_eps) * (which == 0 ? A.q_scale : 1.f);
        const int brow = which == 0 ? NMAX + i : i;
        uint32_t wh[4], wl[4];
        float kv[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          split_bf16x2(scale * v8[2 * e], scale * v8[2 * e + 1], wh[e], wl[e]);
          kv[2 * e] = __uint_as_float(wh[e] << 16) + __uint_as_float(wl[e] << 16);
          kv[2 * e + 1] =
              __uint_as_float(wh[e] & 0xffff0000u) + __uint_as_float(wl[e] & 0xffff0000u);
        }
        *reinterpret_cast<uint4 *>(B1 + sw128_bf16(R1, brow, li * 8)) =
            make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(B1 + sw128_bf16(R1, NC + brow, li * 8)) =
            make_uint4(wl[0], wl[1], wl[2], wl[3]);
        float4 *kd = reinterpret_cast<float4 *>(kqf + brow * kTcD + li * 8);
        kd[0] = make_float4(kv[0], kv[1], kv[2], kv[3]);
        kd[1] = make_float4(kv[4], kv[5], kv[6], kv[7]);
      }
    }
    // padding rows of this half of the operand are zero
    for (int idx = tid; idx < (NMAX - N) * 16; idx += NT) {
      const int brow = (which == 0 ? NMAX : 0) + N + idx / 16;
      *reinterpret_cast<uint4 *>(B1 + sw128_bf16(R1, brow, 8 * (idx % 16))) =
          make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4 *>(B1 + sw128_bf16(R1, NC + brow, 8 * (idx % 16))) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  {
    // new conv window of the key head's q (threads 0..127) and k (128..255)
    // channels, from the staged old window and inputs
    const int which = tid >> 7, c = tid & (kTcD - 1);
    const unsigned char *cs = which == 0 ? sq : sk;
    const uint16_t *xs = reinterpret_cast<const uint16_t *>(cs + CS::x);
    const float *cc = reinterpret_cast<const float *>(cs + CS::c);
    float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
    const int gc = (which * Hk + kh) * kTcD + c;
    for (int rr = 0; rr < K - 1; ++rr) {
      const int w = crow[rr];
      cache_o[(size_t)rr * C + gc] = w >= 0 ? bf2f(xs[w * kTcD + c]) : cc[(-1 - w) * kTcD + c];
    }
  }
  __syncthreads();
  {
    // Gram entries, 8 threads per item: the parent-path pairs, then the
    // diagonals
    const int items = npair + N;
    const int sub = tid & 7;
    for (int base = 0; base < items; base += NT / 8) {
      const int item = base + (tid >> 3);
      const bool act = item < items;
      int j = 0, n = 0;
      if (act) {
        if (item < npair) {
          j = pj[item];
          n = pn[item];
        } else {
          j = n = item - npair;
        }
      }
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int k = 4 * (sub + 8 * c);
        const float4 kj = *reinterpret_cast<const float4 *>(kqf + j * kTcD + k);
        const float4 kn = *reinterpret_cast<const float4 *>(kqf + n * kTcD + k);
        const float4 qn = *reinterpret_cast<const float4 *>(kqf + (NMAX + n) * kTcD + k);
        s1 += dot4(kj, kn);
        s2 += dot4(kj, qn);
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      }
      if (act && sub == 0) {
        if (item < npair) {
          gkk[item] = s1;
          gkq[item] = s2;
        } else {
          kqn[j] = s2;
        }
      }
    }
  }
  __syncthreads();
  {
    // record -> workspace (and the request's tables, once per request)
    uint4 *rec = reinterpret_cast<uint4 *>(T.ws + tc_tab_bytes<NMAX>(Bq) +
                                           (size_t)g * Ly::rec_bytes);
    for (int i = tid; i < Ly::kB / 16; i += NT) rec[i] = reinterpret_cast<const uint4 *>(B1)[i];
    for (int i = tid; i < GL::bytes / 16; i += NT)
      rec[Ly::kB / 16 + i] = reinterpret_cast<const uint4 *>(smem + PL::gr)[i];
    if (l == 0 && kh == 0) {
      uint4 *tab = reinterpret_cast<uint4 *>(T.ws + (size_t)bq * TL::bytes);
      for (int i = tid; i < TL::bytes / 16; i += NT) tab[i] = reinterpret_cast<const uint4 *>(tb)[i];
    }
  }
}

}  // namespace lbx
