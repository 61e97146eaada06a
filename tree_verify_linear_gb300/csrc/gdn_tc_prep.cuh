// gdn_tc_prep.cuh -- per-key-head preparation for the tensor-core step.
//
// One CTA per (layer l, request b, key head) computes what the step kernel's
// tiles share, so that a tile is only the row work on its state slab:
//   * the q and k conv + SiLU + L2 normalisation along each node's ancestor
//     path (q scaled), written to the workspace as the bf16 hi / lo [K|Q]
//     operand image of the step kernel;
//   * the Gram entries k_j.k_n, k_j.q_n of every (node n, strict ancestor j)
//     pair and k_n.q_n, in fp32 (the tensor cores see hi + lo, within
//     2^-17 of the same values);
//   * for each value head of the key head: its gates in the new labels, the
//     entries of T = (I + diag(b a) M)^-1 and W = Q T on every (node,
//     ancestor-or-self) lane, gamma of each node's parent, the accepted-path
//     coefficients and gamma of the accepted node (a value-head record);
//   * the new conv window of the key head's q and k channels, persisted in
//     place (this CTA is the only reader and writer of those channels);
//   * by the CTAs of layer 0 and key head 0, the request's tree tables.
#pragma once

#include "gdn_tc.cuh"

namespace lbx {


// Tree tables of one request in the new labels (the accepted path, root
// first, takes labels 0..P-1; the other nodes follow in input order, so
// parents still precede children), built by one warp: lane i holds input
// nodes i and i + 32 (N <= NMAX <= 64), ancestor walks are shuffles.
// Parent indices that break the tree rules (the step kernel reports such a
// batch) are clamped so that no index leaves its table.
template <int NMAX>
__device__ void build_tables_warp(int lane, int N, int K, int acc, const int32_t *par_b,
                                  unsigned char *tb) {
  constexpr int S = (NMAX + 31) / 32;  // nodes per lane
  static_assert(S <= 2, "at most two nodes per lane");
  using TL = TabLayout<NMAX>;
  constexpr unsigned FULL = 0xffffffffu;
  unsigned char *pj = tb + TL::pj, *pn = tb + TL::pn, *ln = tb + TL::ln;
  uint16_t *lofs = reinterpret_cast<uint16_t *>(tb + TL::lofs);
  int *par = reinterpret_cast<int *>(tb + TL::par);
  int *dep = reinterpret_cast<int *>(tb + TL::dep);
  int *off = reinterpret_cast<int *>(tb + TL::off);
  int *off2 = reinterpret_cast<int *>(tb + TL::off2);
  int *win = reinterpret_cast<int *>(tb + TL::win);
  int *n2o = reinterpret_cast<int *>(tb + TL::n2o);
  int *o2n = reinterpret_cast<int *>(tb + TL::o2n);
  int *corder = reinterpret_cast<int *>(tb + TL::corder);
  int *crow = reinterpret_cast<int *>(tb + TL::crow);
  int *meta = reinterpret_cast<int *>(tb + TL::meta);
  // value v[] of node m (held by lane m & 31, slot m >> 5); warp-collective,
  // m in [0, 32 S)
  auto at = [&](const int (&v)[S], int m) {
    int r = __shfl_sync(FULL, v[0], m & 31);
    if constexpr (S > 1) {
      const int r1 = __shfl_sync(FULL, v[1], m & 31);
      if (m >= 32) r = r1;
    }
    return r;
  };
  auto ballot64 = [&](const bool (&c)[S]) {
    unsigned long long m = __ballot_sync(FULL, c[0]);
    if constexpr (S > 1) m |= (unsigned long long)__ballot_sync(FULL, c[1]) << 32;
    return m;
  };
  int p[S];
  bool real[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    real[s] = i < N;
    p[s] = real[s] ? par_b[i] : -1;
    if (!(p[s] >= 0 && p[s] < i)) p[s] = -1;
  }
  if (!(acc >= 0 && acc < N)) acc = 0;
  // depth: number of strict ancestors
  int d[S];
  {
    int m[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
      d[s] = 0;
      m[s] = p[s];
    }
#pragma unroll 1
    for (int it = 0; it < NMAX; ++it) {
      bool any = false;
#pragma unroll
      for (int s = 0; s < S; ++s) any |= m[s] >= 0;
      if (!__any_sync(FULL, any)) break;
#pragma unroll
      for (int s = 0; s < S; ++s) {
        const int up = at(p, m[s] >= 0 ? m[s] : 0);
        if (m[s] >= 0) {
          ++d[s];
          m[s] = up;
        }
      }
    }
  }
  // the accepted path (acc and its ancestors): the same walk in every lane
  bool onp[S];
#pragma unroll
  for (int s = 0; s < S; ++s) onp[s] = false;
  {
    int c = acc;
#pragma unroll 1
    for (int it = 0; it <= NMAX && c >= 0; ++it) {
#pragma unroll
      for (int s = 0; s < S; ++s) onp[s] |= lane + 32 * s == c;
      c = at(p, c);
    }
  }
  bool cp[S], cr[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    cp[s] = onp[s] && real[s];
    cr[s] = !onp[s] && real[s];
  }
  const unsigned long long pathm = ballot64(cp), restm = ballot64(cr);
  const int P = __popcll(pathm);
  // new label: depth on the path, else after the path in input order
  int nlab[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    nlab[s] = onp[s] ? d[s] : P + __popcll(restm & ((1ull << i) - 1ull));
  }
  int newp_src[S];
#pragma unroll
  for (int s = 0; s < S; ++s) newp_src[s] = at(nlab, p[s] >= 0 ? p[s] : 0);
  // conv window rows (input labels) of each node: itself, then ancestors,
  // then cached rows (-1 - row); taps j >= K and padding nodes read row 0
  int wj[S][4];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    int m = real[s] ? lane + 32 * s : -2, past = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int w = 0;
      if (real[s] && j < K) {
        if (m >= 0) {
          w = m;
        } else {
          ++past;
          w = -1 - (K - 1 - past);
        }
      }
      wj[s][j] = w;
      const int up = at(p, m >= 0 ? m : 0);
      if (real[s] && j < K && m >= 0) m = up;
    }
  }
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    if (real[s]) {
      n2o[nlab[s]] = i;
      o2n[i] = nlab[s];
      par[nlab[s]] = p[s] >= 0 ? newp_src[s] : -1;
      dep[nlab[s]] = d[s];
      *reinterpret_cast<int4 *>(win + 4 * nlab[s]) =
          make_int4(wj[s][0], wj[s][1], wj[s][2], wj[s][3]);
    } else if (i < NMAX) {
      n2o[i] = 0;
      o2n[i] = -1;
      par[i] = -1;
      dep[i] = 0;
      *reinterpret_cast<int4 *>(win + 4 * i) = make_int4(0, 0, 0, 0);
    }
  }
  // new-window sources of the persist: row rr takes the (K-2-rr)-th
  // ancestor of acc, or old cache row depth(acc)+1+rr where the path is short
  {
    const int da = at(d, acc);
    int src[3] = {0, 0, 0};
    int m = acc;
#pragma unroll
    for (int step = 0; step < 3; ++step) {  // m = step-th ancestor of acc
#pragma unroll
      for (int rr = 0; rr < 3; ++rr)
        if (rr < K - 1 && K - 2 - rr == step && step <= da) src[rr] = m;
      m = at(p, m >= 0 ? m : 0);
    }
#pragma unroll
    for (int rr = 0; rr < 3; ++rr)
      if (rr < K - 1 && K - 2 - rr > da) src[rr] = -1 - (da + 1 + rr);
    if (lane == 0) {
      for (int rr = 0; rr < 4; ++rr) crow[rr] = rr < 3 && rr < K - 1 ? src[rr] : 0;
    }
  }
  __syncwarp();
  // parent-path and lane offsets in the new labels (node i = lane + 32 s is
  // now a new label): exclusive prefix sums of depth and depth + 1
  int dl[S], pl[S], e1[S], e2[S];
  int carry1 = 0, carry2 = 0;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    dl[s] = i < N ? dep[i] : 0;
    pl[s] = i < N ? par[i] : -1;
    const int v2 = i < N ? dl[s] + 1 : 0;
    int s1 = dl[s], s2 = v2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t1 = __shfl_up_sync(FULL, s1, o), t2 = __shfl_up_sync(FULL, s2, o);
      if (lane >= o) {
        s1 += t1;
        s2 += t2;
      }
    }
    e1[s] = carry1 + s1 - dl[s];
    e2[s] = carry2 + s2 - v2;
    carry1 += __shfl_sync(FULL, s1, 31);
    carry2 += __shfl_sync(FULL, s2, 31);
  }
  // conv order: nodes whose window lies inside the tree (depth >= K-1) first
  bool ins[S], outs[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    ins[s] = i < N && dl[s] >= K - 1;
    outs[s] = i < N && !ins[s];
  }
  const unsigned long long insm = ballot64(ins), outm = ballot64(outs);
  const int n_inside = __popcll(insm);
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    const unsigned long long lt = (1ull << i) - 1ull;
    if (i < N)
      corder[ins[s] ? __popcll(insm & lt) : n_inside + __popcll(outm & lt)] = i;
    else if (i < NMAX)
      corder[i] = 0;
    if (i <= NMAX) {
      off[i] = e1[s];
      off2[i] = e2[s];
    }
  }
  if (lane == 0) {
    meta[0] = P;
    meta[1] = carry2;  // lanes
    meta[2] = carry1;  // pairs
    meta[3] = n_inside;
  }
  // pairs (node, strict ancestor) and lanes (node, ancestor-or-self)
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = lane + 32 * s;
    int j = pl[s], tt = 0;
    if (i < N) {
      ln[e2[s]] = (unsigned char)i;
      lofs[e2[s]] = (uint16_t)plain_bf16(TcLayout<NMAX>::KP, i, i);
    }
#pragma unroll 1
    for (int it = 0; it < NMAX && __any_sync(FULL, j >= 0); ++it) {
      if (i < N && j >= 0) {
        pj[e1[s] + tt] = (unsigned char)j;
        pn[e1[s] + tt] = (unsigned char)i;
        ln[e2[s] + tt + 1] = (unsigned char)i;
        lofs[e2[s] + tt + 1] = (uint16_t)plain_bf16(TcLayout<NMAX>::KP, i, j);
        ++tt;
      }
      const int up = at(pl, j >= 0 ? j : 0);
      if (j >= 0) j = up;
    }
  }
  __syncwarp();
}

template <int NMAX>
__global__ void __launch_bounds__(TcRes<NMAX>::prep_threads, TcRes<NMAX>::prep_ctas)
    gdn_qk_prep_kernel(const __grid_constant__ TcMaps maps, const TcArgs T) {
  using Ly = TcLayout<NMAX>;
  using PL = PrepLayout<NMAX>;
  using CS = ConvStage<NMAX>;
  using TL = TabLayout<NMAX>;
  using GL = GramLayout<NMAX>;
  using HL = HeadLayout<NMAX>;
  constexpr int kPrepThreads = TcRes<NMAX>::prep_threads;
  constexpr int NT = kPrepThreads, NC = Ly::NC, R1 = Ly::R1, TP = Ly::TP, NP = PL::NP;
  constexpr int kPrepHeads = PL::kPrepHeads;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *sq = smem + PL::sq, *sk = smem + PL::sk;
  float *kqf = reinterpret_cast<float *>(smem + PL::kqf);
  float *gkk = reinterpret_cast<float *>(smem + PL::gr + GL::gkk);
  float *gkq = reinterpret_cast<float *>(smem + PL::gr + GL::gkq);
  float *kqn = reinterpret_cast<float *>(smem + PL::gr + GL::kqn);
  unsigned char *tb = smem + PL::tb;
  int *misc = reinterpret_cast<int *>(smem + PL::misc);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + PL::bar);
  // per-head scratch, in the staging bytes once the conv is done
  float *Tf = reinterpret_cast<float *>(smem + PL::tf);
  float *han = reinterpret_cast<float *>(smem + PL::han);
  float *hbn = reinterpret_cast<float *>(smem + PL::hbn);
  float *hgam = reinterpret_cast<float *>(smem + PL::hgam);
  const int tid = threadIdx.x;
  const int N = A.N, K = A.K, Hk = A.Hk, Hv = A.Hv, Bq = A.Bq;
  const int G = Hv / Hk;
  const int C = (2 * Hk + Hv) * kTcD;
  const uint32_t stg_bytes =
      (uint32_t)N * kTcD * 2 + (uint32_t)(K - 1) * kTcD * 4 + (uint32_t)kTcD * K * 2;

  // the step kernel may be scheduled as this grid's last CTAs start; it waits
  // for this grid's completion before it reads the workspace
  ptx::launch_dependents();
  const int g = blockIdx.x;
  unsigned char *heads = T.ws + tc_head_offset<NMAX>(A.L, Bq, Hk);
  int *porig = reinterpret_cast<int *>(smem + PL::porig);
  const int warp = tid >> 5;
  const int kh = g % Hk, lbi = g / Hk;
  const int bq = lbi % Bq, l = lbi / Bq;
  unsigned char *img = T.ws + tc_tab_bytes<NMAX>(Bq) + (size_t)g * Ly::kB;

  // The copies only read, so they start before the batch is validated (an
  // out-of-range slot is clamped here; such a batch is rejected below).
  int slot_b = A.slot[bq];
  slot_b = slot_b < 0 ? 0 : (slot_b >= A.n_slots ? A.n_slots - 1 : slot_b);
  if (tid == 0) {
    const int crow0 = (l * A.n_slots + slot_b) * (K - 1);
    misc[0] = 0;
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
  // input parents (clamped to the tree rules, so that every window row is a
  // valid index even for a batch rejected below) and the first value heads'
  // gates, in input labels, while the copies fly
  if (tid < NMAX) {
    int p = tid < N ? A.parent[(size_t)bq * N + tid] : -1;
    if (!(p >= 0 && p < tid)) p = -1;
    porig[tid] = p;
  }
  const int nh0 = G < kPrepHeads ? G : kPrepHeads;
  float ga0 = 0.f, gb0 = 0.f;
  if (tid < kPrepHeads * NP) {
    const int hh = tid / NP, o = tid % NP;
    if (hh < nh0 && o < N) {
      const size_t gi = ((size_t)lbi * N + o) * Hv + kh * G + hh;
      ga0 = bf2f(A.a[gi]);
      gb0 = bf2f(A.b[gi]);
    }
  }
  __syncthreads();

  // Warp 0 builds the request's tree tables and checks the batch while warps
  // 1.. run the q and k conv + SiLU + L2 norm of every node (input labels,
  // windows walked along the parents) into fp32 rows.  In the compact layout
  // the k conv runs first (its staged inputs sit in the q rows) and the
  // accepted node's window is kept aside: its K-1 newest raw inputs become
  // the slot's new conv window, written once the batch is known to be valid,
  // after the staged inputs are gone.
  int code = 0;
  float *nwin = reinterpret_cast<float *>(smem + PL::nw);
  if (warp == 0) {
    build_tables_warp<NMAX>(tid, N, K, A.accepted[bq], A.parent + (size_t)bq * N, tb);
    code = validate_batch(A.parent, A.slot, A.accepted, Bq, N, A.n_slots, false, true, true,
                          tid, 32);
  } else {
    // one verdict per warp (the conv below runs whole-warp shuffles)
    const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar, 0));
    if (!ok) code = LBX_ETIMEOUT;
    constexpr int CT = kPrepThreads - 32;  // conv threads
    constexpr int GQ = kTcD / 8;           // 16 threads per node, 8 channels each
    constexpr int U = (NMAX * GQ + CT - 1) / CT;
    static_assert(CT % GQ == 0, "channel group fixed per thread");
    const int ct = tid - 32, li = ct % GQ;
    const int acc = A.accepted[bq];
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int which = PL::kCompact ? 1 - pass : pass;  // 0: q, 1: k
      if (PL::kCompact && pass == 1) ptx::named_sync(1, CT);  // staged k inputs consumed
      if (!ok) continue;
      const unsigned char *cs = which == 0 ? sq : sk;
      float wsl[8][LBX_MAX_CONV_WIDTH];
      conv_weights8<NMAX>(wsl, K, cs, li * 8);
#pragma unroll
      for (int p = 0; p < U; ++p) {
        const int u = p * CT + ct;
        const bool act = u < N * GQ;
        // warps with no node in this pass skip it (u grows with the lane,
        // so the warp's first lane decides)
        if (__shfl_sync(0xffffffffu, u, 0) >= N * GQ) continue;
        const int o = act ? u / GQ : 0;
        // window rows: the node, then its ancestors; past the root the
        // cached rows, newest first (-1 - row); taps j >= K read row 0
        int wj[4];
        bool inside = act;
        {
          int m = o, past = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            int w = 0;
            if (j < K) {
              if (m >= 0) {
                w = m;
              } else {
                ++past;
                w = -1 - (K - 1 - past);
                inside = false;
              }
            }
            wj[j] = w;
            if (j < K && m >= 0) m = porig[m];
          }
        }
        const int4 w4 = make_int4(wj[0], wj[1], wj[2], wj[3]);
        float v8[8];
        // a warp holds two nodes; the inputs-only path when both windows
        // lie inside the tree
        if (__all_sync(0xffffffffu, inside))
          conv8_staged_tree<NMAX>(v8, w4, wsl, cs, li * 8);
        else
          conv8_staged<NMAX>(v8, w4, wsl, cs, li * 8);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
        for (int sh = GQ / 2; sh > 0; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
        if (act) {
          const float scale = rsqrtf(ss + A.l2_eps) * (which == 0 ? A.q_scale : 1.f);
          float4 *kd = reinterpret_cast<float4 *>(kqf + ((which == 0 ? NMAX : 0) + o) * PL::KQP +
                                                  li * 8);
          kd[0] = make_float4(scale * v8[0], scale * v8[1], scale * v8[2], scale * v8[3]);
          kd[1] = make_float4(scale * v8[4], scale * v8[5], scale * v8[6], scale * v8[7]);
        }
      }
      if (PL::kCompact && ct < GQ && acc >= 0 && acc < N) {
        // the slot's new conv window, oldest row first: row rr is window
        // element K-2-rr of the accepted node (raw inputs, copied exactly)
        int w[LBX_MAX_CONV_WIDTH - 1];
        {
          int m = acc, past = 0;
#pragma unroll
          for (int j = 0; j < LBX_MAX_CONV_WIDTH - 1; ++j) {
            if (m >= 0) {
              w[j] = m;
              m = porig[m];
            } else {
              ++past;
              w[j] = -1 - (K - 1 - past);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr) {
          if (rr >= K - 1) break;
          const int j = K - 2 - rr;
          const int wr = j == 0 ? w[0] : (j == 1 ? w[1] : w[2]);
          float4 *dst = reinterpret_cast<float4 *>(
              nwin + (which * (LBX_MAX_CONV_WIDTH - 1) + rr) * kTcD + ct * 8);
          if (wr >= 0) {
            float xv[8];
            unpack8(*reinterpret_cast<const uint4 *>(cs + CS::x + wr * kTcD * 2 + ct * 16), xv);
            dst[0] = make_float4(xv[0], xv[1], xv[2], xv[3]);
            dst[1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
          } else {
            const float4 *cp =
                reinterpret_cast<const float4 *>(cs + CS::c + (-1 - wr) * kTcD * 4 + ct * 32);
            dst[0] = cp[0];
            dst[1] = cp[1];
          }
        }
      }
    }
  }
  // one barrier: conv rows and tables written, and the block's verdict
  if (code) atomicExch(&misc[0], code);
  if (__syncthreads_or(code != 0)) {
    // an invalid batch is reported by the step kernel; a timeout here
    if (tid == 0) {
      if (misc[0] == LBX_ETIMEOUT && A.status) *A.status = LBX_ETIMEOUT;
      (void)ptx::mbar_wait(bar, 0);  // the copies land before the CTA exits
    }
    return;
  }
  const int *dep = reinterpret_cast<const int *>(tb + TL::dep);
  const int *off = reinterpret_cast<const int *>(tb + TL::off);
  const int *off2 = reinterpret_cast<const int *>(tb + TL::off2);
  const int *n2o = reinterpret_cast<const int *>(tb + TL::n2o);
  const int *o2n = reinterpret_cast<const int *>(tb + TL::o2n);
  const unsigned char *pj = tb + TL::pj, *pn = tb + TL::pn, *ln = tb + TL::ln;
  const int *meta = reinterpret_cast<const int *>(tb + TL::meta);
  const int P = meta[0], nl = meta[1], npair = meta[2];

  // operand image in the new labels (K rows, then Q rows; hi rows, then lo
  // rows NC further): the hi / lo split of the fp32 rows, zero padding rows
  for (int idx = tid; idx < NC * (kTcD / 8); idx += NT) {
    const int brow = idx / (kTcD / 8), c8 = idx % (kTcD / 8);
    const int nlab = brow % NMAX;
    uint32_t wh[4] = {0u, 0u, 0u, 0u}, wl[4] = {0u, 0u, 0u, 0u};
    if (nlab < N) {
      const float4 *src = reinterpret_cast<const float4 *>(
          kqf + ((brow - nlab) + n2o[nlab]) * PL::KQP + c8 * 8);
      const float4 x0 = src[0], x1 = src[1];
      split_bf16x2(x0.x, x0.y, wh[0], wl[0]);
      split_bf16x2(x0.z, x0.w, wh[1], wl[1]);
      split_bf16x2(x1.x, x1.y, wh[2], wl[2]);
      split_bf16x2(x1.z, x1.w, wh[3], wl[3]);
    }
    *reinterpret_cast<uint4 *>(img + sw128_bf16(R1, brow, c8 * 8)) =
        make_uint4(wh[0], wh[1], wh[2], wh[3]);
    *reinterpret_cast<uint4 *>(img + sw128_bf16(R1, NC + brow, c8 * 8)) =
        make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
  if (tid < 2 * kTcD) {
    // new conv window of the key head's q (threads 0..127) and k (128..255)
    // channels: kept aside during the conv (compact layout), else from the
    // staged old window and inputs
    const int which = tid >> 7, c = tid & (kTcD - 1);
    float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
    const int gc = (which * Hk + kh) * kTcD + c;
    if (PL::kCompact) {
      for (int rr = 0; rr < K - 1; ++rr)
        cache_o[(size_t)rr * C + gc] = nwin[(which * (LBX_MAX_CONV_WIDTH - 1) + rr) * kTcD + c];
    } else {
      const int *crow = reinterpret_cast<const int *>(tb + TL::crow);
      const unsigned char *cs = which == 0 ? sq : sk;
      const uint16_t *xs = reinterpret_cast<const uint16_t *>(cs + CS::x);
      const float *cc = reinterpret_cast<const float *>(cs + CS::c);
      for (int rr = 0; rr < K - 1; ++rr) {
        const int w = crow[rr];
        cache_o[(size_t)rr * C + gc] = w >= 0 ? bf2f(xs[w * kTcD + c]) : cc[(-1 - w) * kTcD + c];
      }
    }
  }
  {
    // Gram entries, 8 threads per item: the parent-path pairs, then the
    // diagonals (new labels; the fp32 rows are in input labels)
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
      const int jo = n2o[j], no = n2o[n];
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int k = 4 * (sub + 8 * c);
        const float4 kj = *reinterpret_cast<const float4 *>(kqf + jo * PL::KQP + k);
        const float4 kn = *reinterpret_cast<const float4 *>(kqf + no * PL::KQP + k);
        const float4 qn = *reinterpret_cast<const float4 *>(kqf + (NMAX + no) * PL::KQP + k);
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
  __syncthreads();  // the staged inputs are dead from here on

  // ---- the G value heads of this key head, kPrepHeads at a time ----
#pragma unroll 1
  for (int hc = 0; hc < G; hc += kPrepHeads) {
    const int nh = G - hc < kPrepHeads ? G - hc : kPrepHeads;
    // gates of head hc + hh in the new labels (0 for padding nodes); the
    // first heads' were loaded at the start, in input labels
    if (hc == 0) {
      if (tid < kPrepHeads * NP) {
        const int hh = tid / NP, o = tid % NP;
        const int nlab = o < N ? o2n[o] : o;
        han[hh * NP + nlab] = ga0;
        hbn[hh * NP + nlab] = gb0;
        hgam[tid] = 0.f;
      }
    } else {
      for (int idx = tid; idx < kPrepHeads * NP; idx += NT) {
        const int hh = idx / NP, n = idx % NP;
        float av = 0.f, bv = 0.f;
        if (hh < nh && n < N) {
          const size_t gi = ((size_t)lbi * N + n2o[n]) * Hv + kh * G + hc + hh;
          av = bf2f(A.a[gi]);
          bv = bf2f(A.b[gi]);
        }
        han[idx] = av;
        hbn[idx] = bv;
        hgam[idx] = 0.f;
      }
    }
    __syncthreads();
    // one task per (head, node n, ancestor-or-self m): column m of T along
    // the stretch m -> n of the parent path (positions 0..L), then W[n][m]
    for (int task = tid; task < nh * nl; task += NT) {
      const int hh = task / nl, lane = task - hh * nl;
      const float *an = han + hh * NP, *bn = hbn + hh * NP;
      float *tf = Tf + hh * NMAX * TP;
      const int n = ln[lane];
      const int L = lane - off2[n];
      const int e0 = off[n];
      const int m = L == 0 ? n : pj[e0 + L - 1];
      tf[m * TP + m] = 1.f;
      float xl = 1.f;
      for (int p = 1; p <= L; ++p) {
        const int jp = p == L ? n : pj[e0 + (L - p - 1)];
        const int ep = off[jp];
        float s = 0.f, gp = 1.f;
        for (int q = p - 1; q >= 0; --q) {
          const int e = ep + (p - q - 1);
          const int jq = pj[e];
          s = fmaf(gp * gkk[e], tf[jq * TP + m], s);
          gp *= an[jq];
        }
        xl = -bn[jp] * an[jp] * s;
        tf[jp * TP + m] = xl;
      }
      float s = 0.f, gp = 1.f;
      for (int q = L - 1; q >= 0; --q) {
        const int e = e0 + (L - q - 1);
        const int jq = pj[e];
        s = fmaf(gp * gkq[e], tf[jq * TP + m], s);
        gp *= an[jq];
      }
      float *hrec = reinterpret_cast<float *>(
          heads + ((size_t)lbi * Hv + kh * G + hc + hh) * HL::bytes + HL::tw);
      hrec[lane] = xl;
      hrec[HL::lanes4(nl) + lane] = fmaf(kqn[n], xl, an[n] * s);
      if (L == dep[n]) hgam[hh * NP + n] = gp;  // product of the gates of all ancestors
    }
    __syncthreads();
    // gates, gamma, accepted-path coefficients g(j->acc) (path = labels
    // 0..P-1) and gamma of the accepted node
    for (int idx = tid; idx < nh * NP; idx += NT) {
      const int hh = idx / NP, n = idx % NP;
      const float *an = han + hh * NP;
      unsigned char *hb = heads + ((size_t)lbi * Hv + kh * G + hc + hh) * HL::bytes;
      float c = n < P ? 1.f : 0.f;
      for (int u = n + 1; u < P; ++u) c *= an[u];
      reinterpret_cast<float *>(hb + HL::an)[n] = an[n];
      reinterpret_cast<float *>(hb + HL::bn)[n] = hbn[idx];
      reinterpret_cast<float *>(hb + HL::gam)[n] = hgam[idx];
      reinterpret_cast<float *>(hb + HL::cpa)[n] = c;
      if (n == 0) {
        float4 *ga = reinterpret_cast<float4 *>(hb + HL::gacc);
        *ga = make_float4(hgam[hh * NP + P - 1] * an[P - 1], 0.f, 0.f, 0.f);
      }
    }
    __syncthreads();
  }

  if (l == 0 && kh == 0) {
    // the request's tree tables, once per request
    uint4 *tab = reinterpret_cast<uint4 *>(T.ws + (size_t)bq * TL::bytes);
    for (int i = tid; i < TL::bytes / 16; i += NT) tab[i] = reinterpret_cast<const uint4 *>(tb)[i];
  }
}

}  // namespace lbx
