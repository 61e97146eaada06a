// gdn_chain_tc.cuh -- chunked verify step for long chains on tensor cores
// (sm_103a, d = 128).
//
// A chain of N tokens is the tree whose node i has parent i - 1.  One CTA
// owns one (layer l, request b, value head h) sequence and walks it in chunks
// of kChainC tokens: within a chunk the tokens are a kChainC-node chain whose
// root state S0 is the state after the previous chunk, so the closed form of
// the tree step applies unchanged (T = (I + diag(b a) M)^-1, W = Q T, three
// bf16 hi/lo tensor-core products per chunk, the same TMEM map as the tree
// kernel's 16-node instance).  The running state stays in shared memory (fp32)
// from the first chunk to the last: it is read from HBM once and written once,
// at the accepted token.  What the tree path takes from its prep kernel is
// computed here per chunk, since x and o dominate this workload's bytes: the
// q/k conv (+ SiLU + L2) into the [K|Q] operand, the gates, the Gram entries
// and the T/W lanes of the chunk.  The conv inputs of q/k and of v are staged
// by TMA one chunk ahead: each buffer is reloaded as soon as the chunk's conv
// has read it.
#pragma once

#include "gdn_tc.cuh"

namespace lbx {

constexpr int kChainC = 16;   // tokens per chunk
constexpr int kChainRows = kChainC + LBX_MAX_CONV_WIDTH - 1;  // staged rows: 3 before the chunk

// Staged conv inputs of one 128-channel block for one chunk: raw inputs of
// tokens t0-3 .. t0+C-1 (bf16), the slot's cached rows (fp32, used by the
// first chunk only) and the weights (bf16 [128][K]).
struct ChainStage {
  static constexpr int x = 0;
  static constexpr int c = kChainRows * kTcD * 2;
  static constexpr int w = c + (LBX_MAX_CONV_WIDTH - 1) * kTcD * 4;
  static constexpr int bytes = round_up(w + kTcD * LBX_MAX_CONV_WIDTH * 2, 128);
};

struct ChainLayout {
  using Ly = TcLayout<kChainC>;
  using CS = ChainStage;
  static constexpr int kNPair = kChainC * (kChainC - 1) / 2;
  static constexpr int kNLane = kChainC * (kChainC + 1) / 2;
  static constexpr int TP = Ly::TP;
  static constexpr int stage = 0;                          // running state, fp32
  static constexpr int b1 = stage + (int)kStageBytes;      // [K|Q] hi/lo of the chunk
  static constexpr int b2hi = b1 + Ly::kB;
  static constexpr int b2lo = b2hi + Ly::kB2;
  static constexpr int sqk = round_up(b2lo + Ly::kB2, 128);  // q inputs, then k inputs
  static constexpr int sv = sqk + 2 * CS::bytes;           // v inputs
  static constexpr int tf = sv + CS::bytes;                // float [C][TP] T scratch
  static constexpr int gkk = tf + 4 * kChainC * TP;        // float [kNPair]
  static constexpr int gkq = gkk + 4 * round_up(kNPair, 4);
  static constexpr int kqn = gkq + 4 * round_up(kNPair, 4);
  static constexpr int an = kqn + 4 * kChainC;
  static constexpr int bn = an + 4 * kChainC;
  static constexpr int gam = bn + 4 * kChainC;             // gamma of the previous token
  static constexpr int cpa = gam + 4 * kChainC;            // coefficients g(j -> chunk end)
  static constexpr int cac = cpa + 4 * kChainC;            // coefficients g(j -> accepted)
  // float [C][C] matrices of the chunk: L = diag(b a) M, Q, and the scratch
  // of T = (I + L)^-1 (row-major, some also transposed); tf is one of them
  static constexpr int kMP = kChainC + 4;                  // padded row pitch (banks)
  static constexpr int kMat = 4 * kChainC * kMP;
  static constexpr int lm = cac + 4 * kChainC;
  static constexpr int qm = lm + kMat;
  static constexpr int mx = qm + kMat;                     // three more matrices
  static constexpr int misc = mx + 3 * kMat;
  static constexpr int bars = (misc + 64 + 7) & ~7;        // 7 x uint64
  static constexpr int total = bars + 7 * 8;
  static_assert(total <= kTcMaxSmem, "two CTAs per SM");
  static_assert(TP == kChainC, "tf holds a dense C x C matrix");
  static_assert(sqk % 128 == 0 && sv % 128 == 0 && CS::bytes % 128 == 0, "TMA destinations");
};

struct ChainMaps {
  CUtensorMap state;  // [rows][128] fp32, box {32, 128}, 128-byte swizzle
  CUtensorMap x;      // [L*Bq*N][C] bf16, box {128, kChainRows}
  CUtensorMap cache;  // [L*n_slots*(K-1)][C] fp32, box {128, K-1} (K > 1)
};

// hi + lo of 8 consecutive elements of row `row` of an operand image that keeps
// its hi rows first and its lo rows `nc` rows further.
__device__ __forceinline__ void image_row8(const unsigned char *img, int r1, int nc, int row,
                                           int k, float (&v)[8]) {
  float a[8], b[8];
  unpack8(*reinterpret_cast<const uint4 *>(img + sw128_bf16(r1, row, k)), a);
  unpack8(*reinterpret_cast<const uint4 *>(img + sw128_bf16(r1, nc + row, k)), b);
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = a[e] + b[e];
}

struct ChainArgs {
  StepArgs s;
  int n_seq;  // L * Bq * Hv sequences
};

// Window row of tap j (0 = the token itself) of chunk-local token n: a staged
// input row (>= 0) while the token index stays >= 0, else the slot's cached row
// (-1 - row, oldest row first); taps j >= K read row 0 with weight 0.
__device__ __forceinline__ int chain_win(int t0, int n, int j, int K) {
  if (j >= K) return 0;
  const int t = t0 + n - j;
  return t >= 0 ? (LBX_MAX_CONV_WIDTH - 1) + n - j : -1 - (K - 1 + t);
}

__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
    gdn_chain_tc_kernel(const __grid_constant__ ChainMaps maps, const ChainArgs T) {
  using Ly = TcLayout<kChainC>;
  using CL = ChainLayout;
  using CS = ChainStage;
  constexpr int C = kChainC, NMAX = kChainC, NC = Ly::NC, R1 = Ly::R1, KP = Ly::KP, KH = KP / 2;
  constexpr int NH = C / 2, LB = 8;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *st = smem + CL::stage;
  unsigned char *B1 = smem + CL::b1;
  unsigned char *B2hi = smem + CL::b2hi;
  unsigned char *B2lo = smem + CL::b2lo;
  unsigned char *sq = smem + CL::sqk, *sk = sq + CS::bytes, *sv = smem + CL::sv;
  float *Tf = reinterpret_cast<float *>(smem + CL::tf);
  float *gkk = reinterpret_cast<float *>(smem + CL::gkk);
  float *gkq = reinterpret_cast<float *>(smem + CL::gkq);
  float *kqn = reinterpret_cast<float *>(smem + CL::kqn);
  float *an = reinterpret_cast<float *>(smem + CL::an);
  float *bn = reinterpret_cast<float *>(smem + CL::bn);
  float *gam = reinterpret_cast<float *>(smem + CL::gam);
  float *cpa = reinterpret_cast<float *>(smem + CL::cpa);
  float *cac = reinterpret_cast<float *>(smem + CL::cac);
  float *Lm = reinterpret_cast<float *>(smem + CL::lm);
  float *Qm = reinterpret_cast<float *>(smem + CL::qm);
  float *Mx = reinterpret_cast<float *>(smem + CL::mx);  // three C x C matrices
  int *misc = reinterpret_cast<int *>(smem + CL::misc);
  // misc[0] error flag, [2] last arriver, [3] TMEM base
  float *fmisc = reinterpret_cast<float *>(misc + 8);  // [0] gamma_end, [1] gamma_acc
  uint64_t *stage_bar = reinterpret_cast<uint64_t *>(smem + CL::bars);
  uint64_t *qk_bar = stage_bar + 1;
  uint64_t *v_bar = stage_bar + 2;
  uint64_t *mma_bar = stage_bar + 3;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const bool lead = tid == 0;
  const int N = A.N, K = A.K, Hk = A.Hk, Hv = A.Hv, Bq = A.Bq;
  const int G = Hv / Hk;
  const int Cc = (2 * Hk + Hv) * kTcD;  // conv channels
  const int quad = warp & 3, hf = warp >> 2;
  const int r = quad * 32 + (tid & 31);
  const int n0 = hf * NH;

  {
    int code = validate_batch(A.parent, A.slot, A.accepted, Bq, N, A.n_slots, true, true, true);
    if (ptx::smem_u32(smem) & 1023u) code = LBX_ECUDA;
    code = block_any_error(code, misc);
    if (code) {
      if (tid == 0 && A.status) *A.status = code;
      return;
    }
  }
  if (tid == 0) {
    ptx::mbar_init(stage_bar, 1);
    ptx::mbar_init(qk_bar, 1);
    ptx::mbar_init(v_bar, 1);
    ptx::mbar_init(mma_bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t *>(&misc[3]), kTcTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  // entries of [T|W] above the diagonal stay 0
  for (int idx = tid; idx < 2 * Ly::kB2 / 16; idx += kTcThreads)
    *reinterpret_cast<uint4 *>(B2hi + 16 * idx) = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[3]);
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
  const uint32_t x_bytes = (uint32_t)kChainRows * kTcD * 2;
  const uint32_t c_bytes = (uint32_t)(K - 1) * kTcD * 4;
  const uint32_t w_bytes = (uint32_t)kTcD * K * 2;

  uint32_t stage_waits = 0, qk_waits = 0, v_waits = 0, mma_waits = 0;
  int n_stage = 0, n_qk = 0, n_v = 0;
  // a wait that timed out in this thread (bad); the block's decision to stop
  // (aborted), taken at a barrier reduction so that every thread agrees
  bool bad = false, aborted = false;
  auto wait_on = [&](uint64_t *bar, uint32_t &waits) {
    if (!ptx::mbar_wait(bar, waits & 1u)) {
      if (A.status) *A.status = LBX_ETIMEOUT;
      bad = true;
    }
    ++waits;
  };
  // lead: one chunk's conv inputs of channel block ch0 into dst (the cached
  // rows and the weights with the first chunk only)
  auto stage_block = [&](unsigned char *dst, int ch0, int lbi, int l, int slot_b, int t0,
                         uint64_t *bar) {
    ptx::tma_load_2d(dst + CS::x, &maps.x, ch0, lbi * N + t0 - (LBX_MAX_CONV_WIDTH - 1), bar);
    if (t0 == 0) {
      if (K > 1)
        ptx::tma_load_2d(dst + CS::c, &maps.cache, ch0, (l * A.n_slots + slot_b) * (K - 1), bar);
      ptx::bulk_load(dst + CS::w, A.conv_w + (size_t)l * Cc * K + (size_t)ch0 * K, w_bytes, bar);
    }
  };

  float gna = 0.f, gnb = 0.f;  // gates of token tid (< C) of the next chunk
#pragma unroll 1
  for (int seq = blockIdx.x; seq < T.n_seq; seq += gridDim.x) {
    const int h = seq % Hv, lbi = seq / Hv, bq = lbi % Bq, l = lbi / Bq, kh = h / G;
    const int slot_b = A.slot[bq], acc = A.accepted[bq];
    const int nch = (N + C - 1) / C, ch_acc = acc / C;
    const uint16_t *a_lb = A.a + (size_t)lbi * N * Hv, *b_lb = A.b + (size_t)lbi * N * Hv;
    if (lead) {
      ptx::mbar_arrive_expect_tx(stage_bar, kStageBytes);
      const int srow = ((l * A.n_slots + slot_b) * Hv + h) * kTcD;
      for (int a = 0; a < 4; ++a)
        ptx::tma_load_2d(st + a * (kStageBytes / 4), &maps.state, a * 32, srow, stage_bar);
      ++n_stage;
      ptx::mbar_arrive_expect_tx(qk_bar, 2 * (x_bytes + c_bytes + w_bytes));
      stage_block(sq, kh * kTcD, lbi, l, slot_b, 0, qk_bar);
      stage_block(sk, (Hk + kh) * kTcD, lbi, l, slot_b, 0, qk_bar);
      ++n_qk;
      ptx::mbar_arrive_expect_tx(v_bar, x_bytes + c_bytes + w_bytes);
      stage_block(sv, (2 * Hk + h) * kTcD, lbi, l, slot_b, 0, v_bar);
      ++n_v;
    }
    if (tid < C) {
      gna = tid < N ? bf2f(a_lb[(size_t)tid * Hv + h]) : 0.f;
      gnb = tid < N ? bf2f(b_lb[(size_t)tid * Hv + h]) : 0.f;
    }

#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      const int t0 = ch * C;
      const int nc = N - t0 < C ? N - t0 : C;
      // ---- gates of this chunk (0 on padding tokens); the next chunk's in flight ----
      if (tid < C) {
        an[tid] = tid < nc ? gna : 0.f;
        bn[tid] = tid < nc ? gnb : 0.f;
        if (ch + 1 < nch) {
          const int t = t0 + C + tid;
          gna = t < N ? bf2f(a_lb[(size_t)t * Hv + h]) : 0.f;
          gnb = t < N ? bf2f(b_lb[(size_t)t * Hv + h]) : 0.f;
        }
      }

      // ---- q, k: conv + SiLU + L2 -> [K|Q] operand (padding tokens: 0) ----
      wait_on(qk_bar, qk_waits);
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const unsigned char *cs = which == 0 ? sq : sk;
        constexpr int GQ = kTcD / 8;
        static_assert(C * GQ == kTcThreads, "one (node, 8 channels) unit per thread");
        const int li = tid % GQ, i = tid / GQ;
        float wsl[8][LBX_MAX_CONV_WIDTH];
        conv_weights8<kChainRows>(wsl, K, cs, li * 8);
        const int4 w4 = make_int4(chain_win(t0, i, 0, K), chain_win(t0, i, 1, K),
                                  chain_win(t0, i, 2, K), chain_win(t0, i, 3, K));
        float v8[8];
        if (t0 >= LBX_MAX_CONV_WIDTH - 1)
          conv8_staged_tree<kChainRows>(v8, w4, wsl, cs, li * 8);
        else
          conv8_staged<kChainRows>(v8, w4, wsl, cs, li * 8);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
        for (int o = GQ / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float scale =
            i < nc ? rsqrtf(ss + A.l2_eps) * (which == 0 ? A.q_scale : 1.f) : 0.f;
        const int brow = which == 0 ? NMAX + i : i;
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split_bf16x2(scale * v8[2 * e], scale * v8[2 * e + 1], wh[e], wl[e]);
        *reinterpret_cast<uint4 *>(B1 + sw128_bf16(R1, brow, li * 8)) =
            make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(B1 + sw128_bf16(R1, NC + brow, li * 8)) =
            make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
      ptx::fence_proxy_async();
      __syncthreads();  // operand written; q/k inputs consumed
      if (lead) {
        if (ch + 1 < nch) {
          ptx::mbar_arrive_expect_tx(qk_bar, 2 * x_bytes);
          stage_block(sq, kh * kTcD, lbi, l, slot_b, t0 + C, qk_bar);
          stage_block(sk, (Hk + kh) * kTcD, lbi, l, slot_b, t0 + C, qk_bar);
          ++n_qk;
        }
        if (ch == 0) {
          // the old q/k window of the key head has been read: arrive; the last
          // of the G sequences of the key head writes the new one at its end
          unsigned int *cnt = A.counters + (size_t)lbi * Hk + kh;
          const unsigned int prev = atomicAdd(cnt, 1u);
          misc[2] = prev == (unsigned int)(G - 1);
          if (misc[2]) atomicExch(cnt, 0u);
        }
      }

      // ---- Gram matrix K [K|Q]^T on the tensor cores: the product MMA1
      // forms with S0, taken with the operand's first 32 rows (K, then Q) as
      // A.  Warps 0 and 4 (TMEM lanes 0..31) copy those rows, hi and lo, into
      // the S0 columns, free until the split; lanes 32..127 of A and of the
      // product are not used.  Warp 1 meanwhile forms the gate products: gamma
      // of the previous token, coefficients to the chunk's last token and to
      // the accepted token ----
      const bool acc_here = ch == ch_acc;
      const int acc_l = acc - t0;
      if (warp == 0 || warp == 4) {
        const int lo = warp >> 2, row = lo * NC + (tid & 31);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 u =
                *reinterpret_cast<const uint4 *>(B1 + sw128_bf16(R1, row, 64 * c + 8 * q));
            v[4 * q] = u.x;
            v[4 * q + 1] = u.y;
            v[4 * q + 2] = u.z;
            v[4 * q + 3] = u.w;
          }
          ptx::tmem_st32(tq + Ly::cA1 + 64 * lo + 32 * c, v);
        }
        ptx::tmem_wait_st();
      } else if (warp == 1) {
        // prefix and suffix products of the gates over the chunk's tokens
        const int lane = tid & 31;
        const float a = lane < C ? an[lane] : 1.f;
        float pre = a;  // a_0 ... a_lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, pre, o);
          if (lane >= o) pre *= t;
        }
        const float pre_ex = __shfl_up_sync(0xffffffffu, pre, 1);
        auto suffix_from = [&](int end) {  // product of a_(lane+1) .. a_(end-1)
          float suf = lane < end ? a : 1.f;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf *= t;
          }
          const float ex = __shfl_down_sync(0xffffffffu, suf, 1);
          return lane + 1 < 32 ? ex : 1.f;
        };
        const float c_end = suffix_from(nc);
        const float c_acc = suffix_from(acc_here ? acc_l + 1 : 0);
        const float g_end = __shfl_sync(0xffffffffu, pre, nc - 1);
        const float g_acc = __shfl_sync(0xffffffffu, pre, acc_here ? acc_l : 0);
        if (lane < C) {
          gam[lane] = lane == 0 ? 1.f : pre_ex;
          cpa[lane] = lane < nc ? c_end : 0.f;
          cac[lane] = acc_here && lane <= acc_l ? c_acc : 0.f;
        }
        if (lane == 0) {
          fmisc[0] = g_end;
          fmisc[1] = g_acc;
        }
      }
      ptx::tc_fence_before();
      __syncthreads();
      if (lead) {
        ptx::tc_fence_after();
        mma_kq<NMAX>(tmem + Ly::cD1, tmem + Ly::cA1, ptx::smem_u32(B1));
        ptx::mma_commit(mma_bar);
      }
      wait_on(mma_bar, mma_waits);
      ptx::tc_fence_after();
      if (warp == 0 || warp == 4) {
        // lane j < C: k_j.k_n = column n + column NC + n (warp 0), k_j.q_n =
        // column NMAX + n + column NC + NMAX + n (warp 4)
        const int c0 = warp == 0 ? 0 : NMAX;
        float g0[16], g1[16];
        ptx::tmem_ld16(tq + Ly::cD1 + c0, g0);
        ptx::tmem_ld16(tq + Ly::cD1 + NC + c0, g1);
        ptx::tmem_wait_ld();
        const int jr = tid & 31;
        float *dst = warp == 0 ? gkk : gkq;
        if (jr < C) {
#pragma unroll
          for (int n = 0; n < C; ++n) {
            const float v = g0[n] + g1[n];
            if (n > jr) dst[n * (n - 1) / 2 + (n - 1 - jr)] = v;
            if (warp == 4 && n == jr) kqn[n] = v;
          }
        }
      }
      ptx::tc_fence_before();
      __syncthreads();

      // ---- T = (I + L)^-1 with L = diag(b a) M, and W = Q T, for the
      // chunk's chain: L[n][j] = b_n a_n g(j->n-1) k_j.k_n, Q[n][j] =
      // a_n g(j->n-1) k_j.q_n (j < n), Q[n][n] = k_n.q_n ----
      // C x C products of lower-triangular matrices, one entry (n, m) per
      // thread: row n of X (row-major) times column m of Y (row m of Y^T),
      // four 16-byte loads each; rows MP floats apart (Tf: C)
      const int en = tid >> 4, em = tid & 15;
      constexpr int MP = CL::kMP;
      auto row_dot = [&](const float *X, int xp, const float *YT) {
        const float4 *x4 = reinterpret_cast<const float4 *>(X + en * xp);
        const float4 *y4 = reinterpret_cast<const float4 *>(YT + em * MP);
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < C / 4; ++q) {
          const float4 xa = x4[q], ya = y4[q];
          acc = fmaf(xa.x, ya.x, fmaf(xa.y, ya.y, fmaf(xa.z, ya.z, fmaf(xa.w, ya.w, acc))));
        }
        return acc;
      };
      // matrices: Lm, LmT, Ma, MaT and Tf, reused as the steps go
      float *LmT = Mx, *Ma = Mx + C * MP, *MaT = Mx + 2 * C * MP;
      {
        // entry (n, j): g(j -> n-1) = a_(j+1) ... a_(n-1), a suffix product over
        // the half-warp of row n (lane u holds a_u for u < n, else 1)
        const int n = en, j = em;
        float sfx = j < n ? an[j] : 1.f;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
          const float t = __shfl_down_sync(0xffffffffu, sfx, o, 16);
          if (j + o < 16) sfx *= t;
        }
        const float g_next = __shfl_down_sync(0xffffffffu, sfx, 1, 16);
        const float g = j < 15 ? g_next : 1.f;
        float lv = 0.f, qv = j == n ? kqn[n] : 0.f;
        if (j < n) {
          const int e = n * (n - 1) / 2 + (n - 1 - j);
          lv = bn[n] * an[n] * g * gkk[e];
          qv = an[n] * g * gkq[e];
        }
        Lm[n * MP + j] = lv;
        LmT[j * MP + n] = lv;
        Qm[n * MP + j] = qv;
      }
      __syncthreads();
      // T = (I + L)^-1 = (I - L)(I + L^2)(I + L^4)(I + L^8), since L^16 = 0
      {
        const float l2 = row_dot(Lm, MP, LmT);  // L^2 -> Ma, MaT
        Ma[en * MP + em] = l2;
        MaT[em * MP + en] = l2;
      }
      __syncthreads();
      {
        const float l4 = row_dot(Ma, MP, MaT);  // L^4 -> Lm, LmT
        const float la = row_dot(Lm, MP, MaT);  // L L^2
        const float id = en == em ? 1.f : 0.f;
        const float p = id - Lm[en * MP + em] + Ma[en * MP + em] - la;  // P = (I - L)(I + L^2)
        __syncthreads();  // every read of L and L^2 done
        Tf[en * C + em] = p;
        Lm[en * MP + em] = l4;
        LmT[em * MP + en] = l4;
      }
      __syncthreads();
      {
        const float l8 = row_dot(Lm, MP, LmT);              // L^8
        const float p2 = Tf[en * C + em] + row_dot(Tf, C, LmT);  // P (I + L^4)
        __syncthreads();  // every read of P and L^4 done
        Ma[en * MP + em] = p2;
        MaT[em * MP + en] = l8;
      }
      __syncthreads();
      {
        const float t = Ma[en * MP + em] + row_dot(Ma, MP, MaT);  // P (I + L^4)(I + L^8)
        Tf[en * C + em] = t;                                  // T
        LmT[em * MP + en] = t;                                 // T^T
      }
      __syncthreads();
      {
        // W[n][m] = Q[n] . T[:, m]; T and W entries (n >= m) -> [T|W]
        const int n = en, m = em;
        if (m <= n) {
          const float wv = row_dot(Qm, MP, LmT);
          const float tv = Tf[n * C + m];
          uint16_t th, tl, wh, wl;
          split_bf16(tv, th, tl);
          split_bf16(wv, wh, wl);
          const uint32_t o = plain_bf16(KP, n, m);
          *reinterpret_cast<uint16_t *>(B2hi + o) = th;
          *reinterpret_cast<uint16_t *>(B2lo + o) = tl;
          *reinterpret_cast<uint16_t *>(B2hi + o + Ly::kWOff) = wh;
          *reinterpret_cast<uint16_t *>(B2lo + o + Ly::kWOff) = wl;
        }
      }
      ptx::fence_proxy_async();

      // ---- running state -> tensor memory (bf16 hi / lo), this thread's 64 columns ----
      if (ch == 0) wait_on(stage_bar, stage_waits);
      {
        uint32_t vh[32], vl[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float4 x4 =
              *reinterpret_cast<const float4 *>(st + sw128_f32(kTcD, r, hf * 64 + 4 * q));
          split_bf16x2(x4.x, x4.y, vh[2 * q], vl[2 * q]);
          split_bf16x2(x4.z, x4.w, vh[2 * q + 1], vl[2 * q + 1]);
        }
        ptx::tmem_st32(tq + Ly::cA1 + hf * 32, vh);
        ptx::tmem_st32(tq + Ly::cA1 + 64 + hf * 32, vl);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      if (__syncthreads_or(bad)) {  // ------------------------------------------------ S1
        aborted = true;
        break;
      }
      if (lead) {
        ptx::tc_fence_after();
        mma_kq<NMAX>(tmem + Ly::cD1, tmem + Ly::cA1, ptx::smem_u32(B1));
        ptx::mma_commit(mma_bar);
      }

      // ---- v of this row for this thread's tokens ----
      wait_on(v_bar, v_waits);
      float vv[NH];
      {
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(sv + CS::x);
        const float *cs = reinterpret_cast<const float *>(sv + CS::c);
        const uint16_t *ws = reinterpret_cast<const uint16_t *>(sv + CS::w) + r * K;
        float wslot[LBX_MAX_CONV_WIDTH];
#pragma unroll
        for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j)
          wslot[j] = j < K ? bf2f(ws[K - 1 - j >= 0 ? K - 1 - j : 0]) : 0.f;
        if (t0 >= LBX_MAX_CONV_WIDTH - 1) {
          // past the first chunk every window row is a staged input row
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            float y = 0.f;
#pragma unroll
            for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j)
              y = fmaf(wslot[j], bf2f(xs[chain_win(t0, n0 + i, j, K) * kTcD + r]), y);
            vv[i] = silu_fast(y);
          }
        } else {
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            float y = 0.f;
#pragma unroll
            for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j) {
              const int w = chain_win(t0, n0 + i, j, K);
              const float xn = bf2f(xs[(w >= 0 ? w : 0) * kTcD + r]);
              const float xc = cs[(w >= 0 ? 0 : -1 - w) * kTcD + r];
              y = fmaf(wslot[j], w >= 0 ? xn : xc, y);
            }
            vv[i] = silu_fast(y);
          }
        }
      }
      ptx::named_sync(1, kTcThreads);  // v inputs consumed
      if (lead && ch + 1 < nch) {
        ptx::mbar_arrive_expect_tx(v_bar, x_bytes);
        stage_block(sv, (2 * Hk + h) * kTcD, lbi, l, slot_b, t0 + C, v_bar);
        ++n_v;
      }

      // ---- rhs -> tensor memory ----
      wait_on(mma_bar, mma_waits);
      ptx::tc_fence_after();
      float oq[NH];
      auto rhs_half = [&](auto hfc) {
        constexpr int HF = decltype(hfc)::value;
        constexpr int N0 = HF * NH;
        float k_hi[LB], k_lo[LB], q_hi[LB], q_lo[LB];
        ptx::tmem_ld_w<LB>(tq + Ly::cD1 + N0, k_hi);
        ptx::tmem_ld_w<LB>(tq + Ly::cD1 + NC + N0, k_lo);
        ptx::tmem_ld_w<LB>(tq + Ly::cD1 + NMAX + N0, q_hi);
        ptx::tmem_ld_w<LB>(tq + Ly::cD1 + NC + NMAX + N0, q_lo);
        ptx::tmem_wait_ld();
        float rhs[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) {
          const int n = N0 + i;
          const float ag = an[n] * gam[n];
          rhs[i] = bn[n] * fmaf(-ag, k_hi[i] + k_lo[i], vv[i]);
          oq[i] = ag * (q_hi[i] + q_lo[i]);
        }
        store_pairs<NMAX, HF>(tq + Ly::cA2, rhs);
      };
      if (hf == 0)
        rhs_half(std::integral_constant<int, 0>{});
      else
        rhs_half(std::integral_constant<int, 1>{});
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      if (__syncthreads_or(bad)) {  // ------------------------------------------------ S2
        aborted = true;
        break;
      }
      if (lead) {
        // MMA2: [delta | W rhs] = rhs [T|W]^T, three passes over K = KP
        ptx::tc_fence_after();
        constexpr uint32_t idesc = ptx::idesc_bf16(128, NC);
        const uint32_t b2h = ptx::smem_u32(B2hi), b2l = ptx::smem_u32(B2lo);
        uint32_t accum = 0;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t a_col = Ly::cA2 + (pass == 2 ? KH : 0);
          const uint32_t b_base = pass == 1 ? b2l : b2h;
#pragma unroll
          for (int ks = 0; ks < KP / 16; ++ks) {
            ptx::mma_bf16_ts(tmem + Ly::cD2, tmem + a_col + 8 * ks,
                             ptx::sdesc(b_base + 256u * ks, 128u, (uint32_t)KP * 16u, 0u), idesc,
                             accum);
            accum = 1;
          }
        }
        ptx::mma_commit(mma_bar);
      }

      // ---- o, and this thread's deltas ----
      wait_on(mma_bar, mma_waits);
      ptx::tc_fence_after();
      float dd[NH];
      {
        float wr[LB];
        ptx::tmem_ld_w<LB>(tq + Ly::cD2 + n0, dd);
        ptx::tmem_ld_w<LB>(tq + Ly::cD2 + NMAX + n0, wr);
        ptx::tmem_wait_ld();
        float *o_base = A.o + ((size_t)lbi * N + t0) * Hv * kTcD + (size_t)h * kTcD + r;
#pragma unroll
        for (int i = 0; i < NH; ++i)
          if (n0 + i < nc) __stcs(o_base + (size_t)(n0 + i) * Hv * kTcD, oq[i] + wr[i]);
      }

      // ---- state passes: g S0 + sum_j coef_j delta_j k_j^T (MMA3) to the
      // accepted token (-> global memory) and to the chunk's last token (->
      // the running state in shared memory) ----
      auto state_pass = [&](const float *coef, float g, bool to_global, bool to_stage) {
        float dl[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) dl[i] = coef[n0 + i] * dd[i];
        if (hf == 0)
          store_pairs<NMAX, 0>(tq + Ly::cA2, dl);
        else
          store_pairs<NMAX, 1>(tq + Ly::cA2, dl);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int k0 = 64 * hf + 32 * c;
          uint32_t gs[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 s4 =
                *reinterpret_cast<const float4 *>(st + sw128_f32(kTcD, r, k0 + 4 * q));
            gs[4 * q] = __float_as_uint(g * s4.x);
            gs[4 * q + 1] = __float_as_uint(g * s4.y);
            gs[4 * q + 2] = __float_as_uint(g * s4.z);
            gs[4 * q + 3] = __float_as_uint(g * s4.w);
          }
          ptx::tmem_st32(tq + Ly::cA1 + k0, gs);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncthreads();
        if (lead) {
          ptx::tc_fence_after();
          constexpr uint32_t idesc = ptx::idesc_bf16_bmn(128, kTcD);
          const uint32_t b1_a = ptx::smem_u32(B1);
#pragma unroll 1
          for (int pass = 0; pass < 3; ++pass) {
            const uint32_t a_col = Ly::cA2 + (pass == 2 ? KH : 0);
            const uint32_t b_base = b1_a + (pass == 1 ? (uint32_t)NC * 128u : 0u);
#pragma unroll
            for (int ks = 0; ks < KP / 16; ++ks)
              ptx::mma_bf16_ts(tmem + Ly::cA1, tmem + a_col + 8 * ks,
                               ptx::sdesc(b_base + 2048u * ks, (uint32_t)R1 * 128u, 1024u, 2u),
                               idesc, 1u);
          }
          ptx::mma_commit(mma_bar);
        }
        wait_on(mma_bar, mma_waits);
        ptx::tc_fence_after();
        float *srow =
            A.state_out + ((((size_t)l * A.n_slots + slot_b) * Hv + h) * kTcD + r) * kTcD;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int k0 = 64 * hf + 32 * c;
          float d[32];
          ptx::tmem_ld32(tq + Ly::cA1 + k0, d);
          ptx::tmem_wait_ld();
          // 16-byte stores: the state is only required to be 16-byte aligned
          if (to_global)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              stg_f4(srow + k0 + 4 * q, make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]));
          if (to_stage)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4 *>(st + sw128_f32(kTcD, r, k0 + 4 * q)) =
                  make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
        }
        ptx::tc_fence_before();
        __syncthreads();
      };
      const bool end_is_acc = acc_here && acc_l == nc - 1;
      if (acc_here && !end_is_acc) state_pass(cac, fmisc[1], true, false);
      if (ch + 1 < nch || end_is_acc) state_pass(cpa, fmisc[0], end_is_acc, ch + 1 < nch);
      __syncthreads();  // the chunk's shared data is free
    }
    if (aborted) break;

    // ---- new conv window of the slot: the K-1 raw inputs ending at the
    // accepted token (continuing into the old window); v channels of this
    // head here, q/k channels of the key head by its last sequence to arrive ----
    {
      const uint16_t *x_lb = A.x + (size_t)lbi * N * Cc;
      const float *cache_s = A.conv_cache + ((size_t)l * A.n_slots + slot_b) * (K - 1) * Cc;
      float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * Cc;
      int src[LBX_MAX_CONV_WIDTH - 1];
#pragma unroll
      for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr) {
        const int t = acc - (K - 2 - rr);
        src[rr] = t >= 0 ? t : -1 - (K - 1 + t);
      }
      if (hf == 0) persist_channel_global((2 * Hk + h) * kTcD + r, K, Cc, src, x_lb, cache_s, cache_o);
      if (misc[2])
        persist_channel_global((hf * Hk + kh) * kTcD + r, K, Cc, src, x_lb, cache_s, cache_o);
    }
    __syncthreads();
  }

  // ---- drain: copies still in flight after an abort ----
  if (lead && aborted) {
    if (n_stage > 0) (void)ptx::mbar_wait(stage_bar, (uint32_t)((n_stage - 1) & 1));
    if (n_qk > 0) (void)ptx::mbar_wait(qk_bar, (uint32_t)((n_qk - 1) & 1));
    if (n_v > 0) (void)ptx::mbar_wait(v_bar, (uint32_t)((n_v - 1) & 1));
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace lbx
