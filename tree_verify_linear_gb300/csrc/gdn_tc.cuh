// gdn_tc.cuh -- fused tree-verify step on tensor cores (sm_103a, d = 128).
//
// Persistent kernel, one CTA per SM: 8 warps, two per TMEM lane quadrant,
// splitting the 128 state columns; single lanes also issue the TMA copies
// (thread 0) and the MMAs (thread 224).  The work is a list of tiles, one per (layer l,
// request b, value head h) = one 128 x 128 fp32 state slab, ordered (l, b,
// key head, head in group); every CTA takes a contiguous range, so consecutive
// tiles usually share their key head and the q/k prologue is computed once
// per key head per CTA.
//
// Everything a tile reads from global memory arrives by bulk-async copies
// issued one tile ahead, on the stage's mbarrier: the state slab S0 (TMA,
// four 32-column boxes, 128-byte swizzle, double-buffered), the raw inputs,
// cached window rows and conv weights of the value head's channels
// (double-buffered), and, when the next tile starts a new key head, those of
// its q and k channels.  Per tile:
//   * the row threads split S0 into bf16 hi + lo parts in tensor memory
//     (operand A, lane = state row);
//   * [k_0..k_{N-1} | q_0..q_{N-1}] (bf16 hi + lo, K-major, 128-byte swizzle)
//     is operand B; three MMAs per K step (hi*hi + hi*lo + lo*hi, relative
//     error ~2^-17) give S0 k_n and S0 q_n for every node in a TMEM
//     accumulator;
//   * the gated delta rule in closed form: with rhs_n = b_n v_n -
//     b_n a_n gamma_p(n) S0 k_n, the deltas of a row are delta = T rhs where
//     T = (I + diag(b a) M)^-1, M[n][j] = g(j->p(n)) k_j.k_n on the parent
//     path (g = product of the gates strictly below j), and
//     o = diag(a gamma) S0 q + W rhs with W = Q T, Q[n][j] = a_n g(j->p(n))
//     k_j.q_n, Q[n][n] = k_n.q_n.  T and W are shared by the 128 rows and
//     built level by level of the tree while the MMAs run;
//   * the accepted state gamma_acc S0 + sum_{j in path(acc)} g(j->acc)
//     delta_j k_j^T overwrites S0 in shared memory and goes back in place by
//     TMA store.
// The conv window of the slot is persisted in place: every value channel by
// its row thread, and the q/k channels, by the CTA whose tile is the last of
// its key-head group to arrive (arrival counter).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "gdn_common.cuh"
#include "gdn_step.cuh"
#include "tc_ptx.cuh"

namespace lbx {

constexpr int kTcD = 128;                       // head dimension of this kernel
constexpr int kTcRowThreads = 256;              // 8 warps: two per TMEM lane quadrant
constexpr int kTcThreads = kTcRowThreads;
constexpr int kTcLoadThread = 0;                // issues the TMA copies
constexpr int kTcMmaThread = 224;               // issues the MMAs
constexpr int kTcArriveThread = 192;            // arrival counter
constexpr uint32_t kTcTmemCols = 256;
constexpr int kTcAHi = 0, kTcALo = 64, kTcD0 = 128;  // TMEM columns (A holds bf16 pairs)
constexpr uint32_t kStageBytes = kTcD * kTcD * 4;    // one state slab, 64 KB
constexpr int kTcMaxSmem = 227 * 1024;

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Staged conv inputs of one 128-channel block for N nodes: raw inputs
// x[n][128] bf16, cached rows [K-1][128] fp32 (oldest first), weights
// [128][K] bf16.
template <int NMAX>
struct ConvStage {
  static constexpr int x = 0;
  static constexpr int c = NMAX * kTcD * 2;
  static constexpr int w = c + (LBX_MAX_CONV_WIDTH - 1) * kTcD * 4;
  static constexpr int bytes = round_up(w + kTcD * LBX_MAX_CONV_WIDTH * 2, 128);
};

template <int NMAX>
struct TcLayout {
  using CS = ConvStage<NMAX>;
  static constexpr int NC = 2 * NMAX;               // B rows / accumulator columns
  static constexpr int kB = NC * kTcD * 2;          // one of B hi / B lo (bf16)
  static constexpr int kNPair = NMAX * (NMAX - 1) / 2 + 1;
  static constexpr int TP = (NMAX + 3) & ~3;        // row pitch of T and W
  static constexpr int stage0 = 0;
  static constexpr int stage1 = stage0 + (int)kStageBytes;
  static constexpr int bhi = stage1 + (int)kStageBytes;
  static constexpr int blo = bhi + kB;
  static constexpr int kf = blo + kB;               // [NMAX][128] fp32 k rows
  static constexpr int tm = kf + NMAX * kTcD * 4;   // [NMAX][TP] T
  static constexpr int wm = tm + NMAX * TP * 4;     // [NMAX][TP] W
  static constexpr int sv0 = round_up(wm + NMAX * TP * 4, 128);  // value-head inputs, 2 slots
  static constexpr int sv1 = sv0 + CS::bytes;
  static constexpr int sq = sv1 + CS::bytes;        // q inputs of the key head
  static constexpr int sk = sq + CS::bytes;         // k inputs of the key head
  static constexpr int pj = sk + CS::bytes;         // int   [kNPair] parent-path nodes
  static constexpr int gkk = pj + 4 * kNPair;       // float [kNPair] k_j . k_n
  static constexpr int gkq = gkk + 4 * kNPair;      // float [kNPair] k_j . q_n
  static constexpr int ckk = gkq + 4 * kNPair;      // float [kNPair] g(j->p) k_j . k_n
  static constexpr int ckq = ckk + 4 * kNPair;      // float [kNPair] g(j->p) k_j . q_n
  static constexpr int par = ckq + 4 * kNPair;
  static constexpr int off = par + 4 * NMAX;        // [NMAX + 4]
  static constexpr int win = off + 4 * (NMAX + 4);  // [NMAX][4]
  static constexpr int lvn = win + 16 * NMAX;       // nodes ordered by depth
  static constexpr int lvo = lvn + 4 * NMAX;        // [NMAX + 4] level starts
  static constexpr int an = lvo + 4 * (NMAX + 4);
  static constexpr int bn = an + 4 * NMAX;
  static constexpr int gam = bn + 4 * NMAX;
  static constexpr int kqn = gam + 4 * NMAX;
  static constexpr int tj = kqn + 4 * NMAX;         // accepted path nodes
  static constexpr int tg = tj + 4 * NMAX;          // and their coefficients
  static constexpr int crow = tg + 4 * NMAX;        // [4] new-window sources (row threads)
  static constexpr int misc = crow + 16;            // ints, see kernel
  static constexpr int bars = (misc + 64 + 7) & ~7; // 3 x uint64
  static constexpr int total = bars + 3 * 8;
  static_assert(kB % 1024 == 0, "operand B must keep 1024-byte alignment");
  static_assert(total <= kTcMaxSmem, "shared memory");
};

struct TcArgs {
  StepArgs s;
  int n_tiles;  // L * Bq * Hv
};

// Byte offset of fp32 element (row, k) of a 128-column slab staged by TMA in
// 32-column boxes with 128-byte swizzle: four atoms of rows x 128 bytes,
// 16-byte chunk index XOR (row & 7).
__device__ __forceinline__ uint32_t sw128_f32(int rows, int row, int k) {
  const int atom = k >> 5, chunk = (k >> 2) & 7;
  return (uint32_t)(atom * rows * 128 + row * 128 + ((chunk ^ (row & 7)) << 4) + ((k & 3) << 2));
}
// Byte offset of bf16 element (row, k) of a K-major operand with 128 bf16
// per row and 128-byte swizzle: two atoms of rows x 128 bytes.
__device__ __forceinline__ uint32_t sw128_bf16(int rows, int row, int k) {
  const int atom = k >> 6, chunk = (k >> 3) & 7;
  return (uint32_t)(atom * rows * 128 + row * 128 + ((chunk ^ (row & 7)) << 4) + ((k & 7) << 1));
}

// bf16 hi / lo split of x: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float x, uint16_t &hi, uint16_t &lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Conv-window sources of the persist: new row rr takes the (K-2-rr)-th
// ancestor of acc, or old cache row depth(acc)+1+rr where the path is short.
__device__ __forceinline__ void window_sources(int *dst, int K, int acc, const int32_t *par_b) {
  int da = 0;
  for (int m = acc; m > 0; m = par_b[m]) ++da;
  for (int rr = 0; rr < K - 1; ++rr) {
    const int dist = K - 2 - rr;
    int w;
    if (dist <= da) {
      int m = acc;
      for (int q = 0; q < dist; ++q) m = par_b[m];
      w = m;
    } else {
      w = -1 - (da + 1 + rr);
    }
    dst[rr] = w;
  }
}

// Conv + SiLU of 8 consecutive channels c0..c0+7 (within a staged block) of
// one node whose window rows are win[0..4) (>= 0: staged x row; < 0: staged
// cache row -1-w; taps j >= K carry weight 0).  Tap K-1 multiplies the node.
// Loads use clamped, always-valid indices and the choice between the node
// row and the cache row is a select, so the unrolled body has no branches.
template <int NMAX>
__device__ __forceinline__ void conv8_staged(float (&out)[8], const int *win, int K,
                                             const unsigned char *cs, int c0) {
  using CS = ConvStage<NMAX>;
  const uint16_t *ws = reinterpret_cast<const uint16_t *>(cs + CS::w);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
  for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j) {
    const int row = win[j];
    const int xr = row >= 0 ? row : 0;
    const int cr = row >= 0 ? 0 : -1 - row;
    float xn[8];
    unpack8(*reinterpret_cast<const uint4 *>(cs + CS::x + xr * kTcD * 2 + c0 * 2), xn);
    const float4 *cp = reinterpret_cast<const float4 *>(cs + CS::c + cr * kTcD * 4 + c0 * 4);
    const float4 lo = cp[0], hi = cp[1];
    const float xc[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const int tap = K - 1 - j >= 0 ? K - 1 - j : 0;
    const float on = j < K ? 1.f : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float wv = on * bf2f(ws[(c0 + e) * K + tap]);
      acc[e] = fmaf(wv, row >= 0 ? xn[e] : xc[e], acc[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) out[e] = silu(acc[e]);
}

// New conv-window entries of staged channel c (global channel gc): row rr
// takes src[rr] (>= 0: staged x row; < 0: staged old cache row -1-src).
template <int NMAX>
__device__ __forceinline__ void persist_staged(const unsigned char *cs, int c, int gc, int K,
                                               int C, const int *src, float *cache_out) {
  using CS = ConvStage<NMAX>;
#pragma unroll
  for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr)
    if (rr < K - 1) {
      const int w = src[rr];
      const float v =
          w >= 0 ? bf2f(reinterpret_cast<const uint16_t *>(cs + CS::x)[w * kTcD + c])
                 : reinterpret_cast<const float *>(cs + CS::c)[(-1 - w) * kTcD + c];
      cache_out[(size_t)rr * C + gc] = v;
    }
}

struct TcMaps {
  CUtensorMap state;  // [rows][128] fp32, box {32, 128}, 128-byte swizzle
  CUtensorMap x;      // [L*Bq*N][C] bf16, box {128, N}
  CUtensorMap cache;  // [L*n_slots*(K-1)][C] fp32, box {128, K-1} (K > 1)
};

template <int NMAX>
__global__ void __launch_bounds__(kTcThreads, 1)
    gdn_step_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs T) {
  using Ly = TcLayout<NMAX>;
  using CS = ConvStage<NMAX>;
  constexpr int NC = Ly::NC;
  constexpr int TP = Ly::TP;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *stage[2] = {smem + Ly::stage0, smem + Ly::stage1};
  unsigned char *svs[2] = {smem + Ly::sv0, smem + Ly::sv1};
  unsigned char *sqs = smem + Ly::sq;
  unsigned char *sks = smem + Ly::sk;
  unsigned char *Bhi = smem + Ly::bhi;
  unsigned char *Blo = smem + Ly::blo;
  float *Kf = reinterpret_cast<float *>(smem + Ly::kf);
  float *Tm = reinterpret_cast<float *>(smem + Ly::tm);
  float *Wm = reinterpret_cast<float *>(smem + Ly::wm);
  int *pj = reinterpret_cast<int *>(smem + Ly::pj);
  float *gkk = reinterpret_cast<float *>(smem + Ly::gkk);
  float *gkq = reinterpret_cast<float *>(smem + Ly::gkq);
  float *ckk = reinterpret_cast<float *>(smem + Ly::ckk);
  float *ckq = reinterpret_cast<float *>(smem + Ly::ckq);
  int *par = reinterpret_cast<int *>(smem + Ly::par);
  int *off = reinterpret_cast<int *>(smem + Ly::off);
  int *win = reinterpret_cast<int *>(smem + Ly::win);
  int *lvn = reinterpret_cast<int *>(smem + Ly::lvn);
  int *lvo = reinterpret_cast<int *>(smem + Ly::lvo);
  float *an = reinterpret_cast<float *>(smem + Ly::an);
  float *bn = reinterpret_cast<float *>(smem + Ly::bn);
  float *gam = reinterpret_cast<float *>(smem + Ly::gam);
  float *kqn = reinterpret_cast<float *>(smem + Ly::kqn);
  int *tj = reinterpret_cast<int *>(smem + Ly::tj);
  float *tg = reinterpret_cast<float *>(smem + Ly::tg);
  int *crow = reinterpret_cast<int *>(smem + Ly::crow);
  int *misc = reinterpret_cast<int *>(smem + Ly::misc);
  // misc[0] error flag, [1] abort, [2] last arriver, [3] TMEM base,
  // [4] accepted-path length, [5] number of tree levels
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + Ly::bars);  // [2]
  uint64_t *mma_bar = full_bar + 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool load_lane = tid == kTcLoadThread;
  const int N = A.N, K = A.K, Hk = A.Hk, Hv = A.Hv, Bq = A.Bq;
  const int G = Hv / Hk;
  const int C = (2 * Hk + Hv) * kTcD;
  const uint32_t x_bytes = (uint32_t)N * kTcD * 2;
  const uint32_t c_bytes = (uint32_t)(K - 1) * kTcD * 4;
  const uint32_t w_bytes = (uint32_t)kTcD * K * 2;

  // ---- whole-batch validation (identical verdict in every CTA) ----
  {
    int code = validate_batch(A.parent, A.slot, A.accepted, Bq, N, A.n_slots, false, true, true);
    // the swizzled TMA / MMA layouts assume a 1024-byte aligned window
    if (ptx::smem_u32(smem) & 1023u) code = LBX_ECUDA;
    code = block_any_error(code, misc);
    if (code) {
      if (tid == 0 && A.status) *A.status = code;
      return;
    }
  }

  // ---- tile range of this CTA ----
  const int nct = gridDim.x;
  const int t_begin = (int)(((long long)T.n_tiles * blockIdx.x) / nct);
  const int t_end = (int)(((long long)T.n_tiles * (blockIdx.x + 1)) / nct);
  const int count = t_end - t_begin;

  // ---- set-up: barriers, TMEM ----
  if (tid == 0) {
    misc[1] = 0;
    ptx::mbar_init(&full_bar[0], 1);
    ptx::mbar_init(&full_bar[1], 1);
    ptx::mbar_init(mma_bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t *>(&misc[3]), kTcTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[3]);

  // Issue every copy tile t needs into stage slot s (control thread): the
  // state slab, the value-head conv inputs and, when `with_qk`, the q/k conv
  // inputs of its key head.
  auto issue_loads = [&](int t, int s, bool with_qk) {
    const int hg = t % G, rest = t / G;
    const int kh = rest % Hk, lbi = rest / Hk;
    const int bq = lbi % Bq, l = lbi / Bq;
    const int h = kh * G + hg;
    const int srow = ((l * A.n_slots + A.slot[bq]) * Hv + h) * kTcD;
    const int xrow = lbi * N;
    const int crow0 = (l * A.n_slots + A.slot[bq]) * (K - 1);
    const uint16_t *w_l = A.conv_w + (size_t)l * C * K;
    const int nblk = with_qk ? 3 : 1;
    const uint32_t bytes = kStageBytes + nblk * (x_bytes + c_bytes + w_bytes);
    ptx::mbar_arrive_expect_tx(&full_bar[s], bytes);
    for (int a = 0; a < 4; ++a)
      ptx::tma_load_2d(stage[s] + a * (kStageBytes / 4), &maps.state, a * 32, srow, &full_bar[s]);
    for (int blk = 0; blk < nblk; ++blk) {
      unsigned char *dst = blk == 0 ? svs[s] : (blk == 1 ? sqs : sks);
      const int ch0 = blk == 0 ? 2 * Hk * kTcD + h * kTcD
                               : (blk == 1 ? kh * kTcD : Hk * kTcD + kh * kTcD);
      ptx::tma_load_2d(dst + CS::x, &maps.x, ch0, xrow, &full_bar[s]);
      if (K > 1) ptx::tma_load_2d(dst + CS::c, &maps.cache, ch0, crow0, &full_bar[s]);
      ptx::bulk_load(dst + CS::w, w_l + (size_t)ch0 * K, w_bytes, &full_bar[s]);
    }
  };

  int pending = -1;          // load thread: stage with an issued, unconsumed load
  uint32_t pending_par = 0;
  if (load_lane && count > 0) {
    issue_loads(t_begin, 0, true);
    pending = 0;
  }

  // row-thread identity: row r (TMEM lane), half hf (column half)
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int hf = (warp >> 2) & 1;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);

  // gates of the current tile, prefetched by threads tid < N
  float ga = 0.f, gb = 0.f;
  if (tid < N && count > 0) {
    const int t = t_begin, hg = t % G, rest = t / G;
    const size_t lbi = (size_t)(rest / Hk);
    const int h = (rest % Hk) * G + hg;
    ga = bf2f(A.a[(lbi * N + tid) * Hv + h]);
    gb = bf2f(A.b[(lbi * N + tid) * Hv + h]);
  }

  int cur_group = -1;
  for (int it = 0; it < count; ++it) {
    const int t = t_begin + it;
    const int s = it & 1;
    const int hg = t % G, rest = t / G;
    const int kh = rest % Hk, lbi = rest / Hk;
    const int bq = lbi % Bq, l = lbi / Bq;
    const int h = kh * G + hg;
    const size_t lb = (size_t)lbi;
    const int slot_b = A.slot[bq];
    float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
    const int32_t *par_b = A.parent + (size_t)bq * N;
    const int acc = A.accepted[bq];
    unsigned char *st = stage[s];
    unsigned char *sv = svs[s];

    {
      // everything this tile reads from global memory
      if (!ptx::mbar_wait(&full_bar[s], (uint32_t)((it >> 1) & 1))) {
        if (A.status) *A.status = LBX_ETIMEOUT;
        atomicExch(&misc[1], 1);
      }
      // ================= group prologue (new key head) =================
      if (rest != cur_group) {
        cur_group = rest;
        for (int i = tid; i < NMAX; i += kTcRowThreads) {
          // conv window rows; taps j >= K and padding nodes point at node 0
          if (i < N) par[i] = par_b[i];
          int m = i < N ? i : -2, past = 0;
          for (int j = 0; j < 4; ++j) {
            int w = 0;
            if (i < N && j < K) {
              if (m >= 0) {
                w = m;
                m = par_b[m];
              } else {
                ++past;
                w = -1 - (K - 1 - past);
              }
            }
            win[i * 4 + j] = w;
          }
        }
        // T and W rows of padding nodes stay zero
        for (int idx = N * TP + tid; idx < NMAX * TP; idx += kTcRowThreads) {
          Tm[idx] = 0.f;
          Wm[idx] = 0.f;
        }
        if (tid == 32) window_sources(crow, K, acc, par_b);
        ptx::named_sync(1, kTcRowThreads);
        if (tid == 0) {
          // depth per node (parents precede children), parent-path offsets,
          // and the nodes grouped by depth
          int dep[NMAX];
          int nlev = 0;
          off[0] = 0;
          for (int i = 0; i < N; ++i) {
            dep[i] = i == 0 ? 0 : dep[par[i]] + 1;
            off[i + 1] = off[i] + dep[i];
            nlev = dep[i] + 1 > nlev ? dep[i] + 1 : nlev;
          }
          int pos = 0;
          for (int d = 0; d < nlev; ++d) {
            lvo[d] = pos;
            for (int i = 0; i < N; ++i)
              if (dep[i] == d) lvn[pos++] = i;
          }
          lvo[nlev] = pos;
          misc[5] = nlev;
        }
        ptx::named_sync(1, kTcRowThreads);
        for (int i = tid; i < N; i += kTcRowThreads) {
          int j = par[i];
          for (int e = off[i]; e < off[i + 1]; ++e) {
            pj[e] = j;
            j = par[j];
          }
        }
        // q/k conv + SiLU + L2 from the staged inputs -> operand B rows
        // (bf16 hi / lo), k rows also in fp32; q scaled
        {
          constexpr int GQ = kTcD / 8;  // 16 threads per (node, q|k)
          constexpr int U = (2 * NMAX * GQ + kTcRowThreads - 1) / kTcRowThreads;
          const int units = 2 * N * GQ;
#pragma unroll
          for (int p = 0; p < U; ++p) {
            const int u = p * kTcRowThreads + tid;
            const bool act = u < units;
            const int grp = act ? u / GQ : 0, li = u % GQ;
            const bool is_q = grp >= N;
            const int i = is_q ? grp - N : grp;
            float v8[8];
            if (act) {
              conv8_staged<NMAX>(v8, win + i * 4, K, is_q ? sqs : sks, li * 8);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[e] = 0.f;
            }
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
            for (int o = GQ / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (act) {
              const float scale = rsqrtf(ss + A.l2_eps) * (is_q ? A.q_scale : 1.f);
              const int brow = is_q ? NMAX + i : i;
              float vv[8];
              uint32_t wh[4], wl[4];
#pragma unroll
              for (int e = 0; e < 8; ++e) vv[e] = scale * v8[e];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                uint16_t h0, l0, h1, l1;
                split_bf16(vv[2 * e], h0, l0);
                split_bf16(vv[2 * e + 1], h1, l1);
                wh[e] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                wl[e] = (uint32_t)l0 | ((uint32_t)l1 << 16);
              }
              const uint32_t o = sw128_bf16(NC, brow, li * 8);
              *reinterpret_cast<uint4 *>(Bhi + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
              *reinterpret_cast<uint4 *>(Blo + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
              if (!is_q) {
                float4 *kd = reinterpret_cast<float4 *>(Kf + i * kTcD + li * 8);
                kd[0] = make_float4(vv[0], vv[1], vv[2], vv[3]);
                kd[1] = make_float4(vv[4], vv[5], vv[6], vv[7]);
              }
            }
          }
          // zero the unused rows of operand B
          const int pad_rows = 2 * (NMAX - N);
          for (int idx = tid; idx < pad_rows * 16; idx += kTcRowThreads) {
            const int pr = idx / 16, q = idx % 16;
            const int brow = pr < NMAX - N ? N + pr : NMAX + N + (pr - (NMAX - N));
            const uint32_t o = sw128_bf16(NC, brow, 8 * q);
            *reinterpret_cast<uint4 *>(Bhi + o) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(Blo + o) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::fence_proxy_async();
        ptx::named_sync(1, kTcRowThreads);
        // Gram entries, 8 threads per item: the parent-path pairs (k_j.k_n
        // and k_j.q_n for j = pj[e]) followed by the N diagonals k_n.q_n
        {
          const int npair = off[N];
          const int items = npair + N;
          const int sub = tid & 7;
          for (int base = 0; base < items; base += kTcRowThreads / 8) {
            const int item = base + (tid >> 3);
            const bool act = item < items;
            int j = 0, n = 0;
            if (act) {
              if (item < npair) {
                j = pj[item];
                while (off[n + 1] <= item) ++n;
              } else {
                j = n = item - npair;
              }
            }
            float s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int k = 8 * (sub + 8 * c);  // 8 consecutive elements
              const float4 *kj = reinterpret_cast<const float4 *>(Kf + j * kTcD + k);
              const float4 *kn = reinterpret_cast<const float4 *>(Kf + n * kTcD + k);
              const uint4 qh = *reinterpret_cast<const uint4 *>(Bhi + sw128_bf16(NC, NMAX + n, k));
              const uint4 ql = *reinterpret_cast<const uint4 *>(Blo + sw128_bf16(NC, NMAX + n, k));
              const uint32_t hw[4] = {qh.x, qh.y, qh.z, qh.w}, lw[4] = {ql.x, ql.y, ql.z, ql.w};
              float qv[8];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                qv[2 * e] = bf16_bits_to_f32(hw[e] & 0xffffu) + bf16_bits_to_f32(lw[e] & 0xffffu);
                qv[2 * e + 1] = bf16_bits_to_f32(hw[e] >> 16) + bf16_bits_to_f32(lw[e] >> 16);
              }
              const float4 j0 = kj[0], j1 = kj[1], n0 = kn[0], n1 = kn[1];
              s1 += dot4(j0, n0) + dot4(j1, n1);
              s2 += dot4(j0, make_float4(qv[0], qv[1], qv[2], qv[3])) +
                    dot4(j1, make_float4(qv[4], qv[5], qv[6], qv[7]));
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
        ptx::named_sync(1, kTcRowThreads);
      }

      // ================= per-tile gates and pair coefficients =================
      if (tid < NMAX) {
        an[tid] = tid < N ? ga : 0.f;
        bn[tid] = tid < N ? gb : 0.f;
        if (tid >= N) gam[tid] = 0.f;
      }
      ptx::named_sync(1, kTcRowThreads);
      for (int i = tid; i < N; i += kTcRowThreads) {
        int j = par[i];
        float g = 1.f;
        for (int e = off[i]; e < off[i + 1]; ++e) {
          ckk[e] = g * gkk[e];
          ckq[e] = g * gkq[e];
          g *= an[j];
          j = par[j];
        }
        gam[i] = g;
      }
      if (tid == 64) {
        // accepted path: acc itself, then its parent path (coefficient g * a_acc)
        int cnt = 0;
        tj[cnt] = acc;
        tg[cnt] = 1.f;
        ++cnt;
        int j = par[acc];
        float g = an[acc];
        while (j >= 0) {
          tj[cnt] = j;
          tg[cnt] = g;
          ++cnt;
          g *= an[j];
          j = par[j];
        }
        misc[4] = cnt;
      }

      // ================= S0 -> tensor memory (bf16 hi / lo) =================
      {
        uint32_t vh[32], vl[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float4 x4 =
              *reinterpret_cast<const float4 *>(st + sw128_f32(kTcD, r, hf * 64 + 4 * q));
          uint16_t h0, l0, h1, l1, h2, l2, h3, l3;
          split_bf16(x4.x, h0, l0);
          split_bf16(x4.y, h1, l1);
          split_bf16(x4.z, h2, l2);
          split_bf16(x4.w, h3, l3);
          vh[2 * q] = (uint32_t)h0 | ((uint32_t)h1 << 16);
          vh[2 * q + 1] = (uint32_t)h2 | ((uint32_t)h3 << 16);
          vl[2 * q] = (uint32_t)l0 | ((uint32_t)l1 << 16);
          vl[2 * q + 1] = (uint32_t)l2 | ((uint32_t)l3 << 16);
        }
        ptx::tmem_st32(tq + kTcAHi + hf * 32, vh);
        ptx::tmem_st32(tq + kTcALo + hf * 32, vl);
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
    }
    __syncthreads();  // ---------------------------------------------- S1
    if (misc[1]) break;

    if (tid == kTcMmaThread) {
      // D = S0 [K|Q]^T: three bf16 passes (hi*hi, hi*lo, lo*hi) over K = 128
      ptx::tc_fence_after();
      constexpr uint32_t idesc = ptx::idesc_bf16(128, NC);
      const uint32_t bhi_a = ptx::smem_u32(Bhi), blo_a = ptx::smem_u32(Blo);
      uint32_t accum = 0;
#pragma unroll 1
      for (int pass = 0; pass < 3; ++pass) {
        const uint32_t a_col = pass == 2 ? kTcALo : kTcAHi;
        const uint32_t b_base = pass == 1 ? blo_a : bhi_a;
#pragma unroll
        for (int ks = 0; ks < kTcD / 16; ++ks) {
          const uint32_t baddr = b_base + (uint32_t)((ks >> 2) * (NC * 128) + (ks & 3) * 32);
          ptx::mma_bf16_ts(tmem + kTcD0, tmem + a_col + 8 * ks, ptx::sdesc_sw128(baddr), idesc,
                           accum);
          accum = 1;
        }
      }
      ptx::mma_commit(mma_bar);
    }
    if (tid == kTcArriveThread) {
      // arrival: this CTA has finished reading the old q/k window of the key
      // head (group prologue, before S1); the last of the G tiles of the
      // group writes the new q/k window
      __threadfence();
      unsigned int *cnt = A.counters + lb * Hk + kh;
      const unsigned int prev = atomicAdd(cnt, 1u);
      const int last = prev == (unsigned int)(G - 1);
      if (last) {
        atomicExch(cnt, 0u);
        __threadfence();
      }
      misc[2] = last;
    }
    if (load_lane) pending = -1;
    __syncwarp();
    {
      // ======== while the MMAs run: T by tree levels, W, this row's v ========
      {
        const int nlev = misc[5];
        for (int d = 0; d < nlev; ++d) {
          for (int idx = lvo[d] + warp; idx < lvo[d + 1]; idx += kTcRowThreads / 32) {
            const int n = lvn[idx];
            if (lane < TP) {
              const float dn = bn[n] * an[n];
              float tv = lane == n ? 1.f : 0.f;
              for (int e = off[n]; e < off[n + 1]; ++e)
                tv = fmaf(-dn * ckk[e], Tm[pj[e] * TP + lane], tv);
              Tm[n * TP + lane] = tv;
            }
          }
          ptx::named_sync(1, kTcRowThreads);
        }
        for (int n = warp; n < N; n += kTcRowThreads / 32) {
          if (lane < TP) {
            const float a_n = an[n];
            float wv = kqn[n] * Tm[n * TP + lane];
            for (int e = off[n]; e < off[n + 1]; ++e)
              wv = fmaf(a_n * ckq[e], Tm[pj[e] * TP + lane], wv);
            Wm[n * TP + lane] = wv;
          }
        }
      }
      // v_n of this row for every node (conv + SiLU of channel r, staged);
      // padding nodes and taps read valid rows with weight 0 / gate 0
      float vv[NMAX];
      {
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(sv + CS::x);
        const float *cs = reinterpret_cast<const float *>(sv + CS::c);
        const uint16_t *ws = reinterpret_cast<const uint16_t *>(sv + CS::w) + r * K;
        float wslot[LBX_MAX_CONV_WIDTH];  // weight of window element j
#pragma unroll
        for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j)
          wslot[j] = j < K ? bf2f(ws[K - 1 - j >= 0 ? K - 1 - j : 0]) : 0.f;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
          float y = 0.f;
#pragma unroll
          for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j) {
            const int w = win[n * 4 + j];
            const float xn = bf2f(xs[(w >= 0 ? w : 0) * kTcD + r]);
            const float xc = cs[(w >= 0 ? 0 : -1 - w) * kTcD + r];
            y = fmaf(wslot[j], w >= 0 ? xn : xc, y);
          }
          vv[n] = silu(y);
        }
      }
      // this row's value channel of the conv window (only this tile reads it)
      if (hf == 0) persist_staged<NMAX>(sv, r, 2 * Hk * kTcD + h * kTcD + r, K, C, crow, cache_o);
      ptx::named_sync(1, kTcRowThreads);
      if (misc[2]) {
        // new q/k window of the key head, from the staged q/k inputs
        const int c = tid & (kTcD - 1);
        if (tid < kTcD) persist_staged<NMAX>(sqs, c, kh * kTcD + c, K, C, crow, cache_o);
        else persist_staged<NMAX>(sks, c, Hk * kTcD + kh * kTcD + c, K, C, crow, cache_o);
      }
      ptx::named_sync(1, kTcRowThreads);
      if (load_lane && it + 1 < count) {
        // next tile's copies, into the other stage once its previous contents
        // (tile it-1) have been read by their TMA store; the staged q/k
        // inputs are free now
        const int s2 = (it + 1) & 1;
        ptx::bulk_wait_read_all();
        issue_loads(t + 1, s2, (t + 1) / G != rest);
        pending = s2;
        pending_par = (uint32_t)(((it + 1) >> 1) & 1);
      }

      // ================= accumulator row -> registers =================
      if (!ptx::mbar_wait(mma_bar, (uint32_t)(it & 1))) {
        if (A.status) *A.status = LBX_ETIMEOUT;
        atomicExch(&misc[1], 1);
      }
      ptx::tc_fence_after();
      float dv[NC];
#pragma unroll
      for (int c = 0; c < NC / 16; ++c) {
        float t16[16];
        ptx::tmem_ld16(tq + kTcD0 + 16 * c, t16);
#pragma unroll
        for (int e = 0; e < 16; ++e) dv[16 * c + e] = t16[e];
      }
      ptx::tmem_wait_ld();

      // rhs_n = b_n v_n - b_n a_n gamma_p S0 k_n ; delta = T rhs ; (hf 1) o
      float rhs[NMAX];  // padding nodes have b = 0, so rhs = 0
#pragma unroll
      for (int n = 0; n < NMAX; ++n) rhs[n] = bn[n] * fmaf(-an[n] * gam[n], dv[n], vv[n]);
      float dl[NMAX];
      {
        float *o_base = A.o + (lb * N) * (size_t)Hv * kTcD + (size_t)h * kTcD + r;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
          float d = 0.f;
#pragma unroll
          for (int m4 = 0; m4 <= n / 4; ++m4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(Tm + n * TP + 4 * m4);
            const float tt[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * m4 + e <= n) d = fmaf(tt[e], rhs[4 * m4 + e], d);
          }
          dl[n] = d;
          if (hf == 1) {
            float ov = an[n] * gam[n] * dv[NMAX + n];
#pragma unroll
            for (int m4 = 0; m4 <= n / 4; ++m4) {
              const float4 w4 = *reinterpret_cast<const float4 *>(Wm + n * TP + 4 * m4);
              const float ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (4 * m4 + e <= n) ov = fmaf(ww[e], rhs[4 * m4 + e], ov);
            }
            if (n < N) __stcs(o_base + (size_t)n * Hv * kTcD, ov);
          }
        }
      }

      // ================= accepted state row, in place (this half) =================
      {
        const int ntgt = misc[4];
        const float gacc = gam[acc] * an[acc];
        float4 accv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)
          accv[q] = f4_scale(gacc, *reinterpret_cast<const float4 *>(
                                       st + sw128_f32(kTcD, r, hf * 64 + 4 * q)));
        for (int m = 0; m < ntgt; ++m) {
          const int j = tj[m];
          float dj = 0.f;
#pragma unroll
          for (int n = 0; n < NMAX; ++n) dj = (j == n) ? dl[n] : dj;
          const float coef = tg[m] * dj;
          const float4 *kr = reinterpret_cast<const float4 *>(Kf + j * kTcD + hf * 64);
#pragma unroll
          for (int q = 0; q < 16; ++q) f4_fma(accv[q], coef, kr[q]);
        }
#pragma unroll
        for (int q = 0; q < 16; ++q)
          *reinterpret_cast<float4 *>(st + sw128_f32(kTcD, r, hf * 64 + 4 * q)) = accv[q];
      }
      // gates of the next tile
      if (tid < N && it + 1 < count) {
        const int t2 = t + 1, hg2 = t2 % G, rest2 = t2 / G;
        const size_t lb2 = (size_t)(rest2 / Hk);
        const int h2 = (rest2 % Hk) * G + hg2;
        ga = bf2f(A.a[(lb2 * N + tid) * Hv + h2]);
        gb = bf2f(A.b[(lb2 * N + tid) * Hv + h2]);
      }
      ptx::fence_proxy_async();
      ptx::tc_fence_before();
    }
    __syncthreads();  // ---------------------------------------------- S3
    if (misc[1]) break;
    if (load_lane) {
      const int row = ((l * A.n_slots + slot_b) * Hv + h) * kTcD;
      for (int a = 0; a < 4; ++a)
        ptx::tma_store_2d(&maps.state, a * 32, row, st + a * (kStageBytes / 4));
      ptx::bulk_commit();
    }
  }

  // ---- drain: an outstanding load (only after an abort) and the stores ----
  if (load_lane) {
    if (pending >= 0 && misc[1]) (void)ptx::mbar_wait(&full_bar[pending], pending_par);
    ptx::bulk_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace lbx
