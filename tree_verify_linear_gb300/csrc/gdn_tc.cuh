// gdn_tc.cuh -- fused tree-verify step on tensor cores (sm_103a, d = 128).
//
// Persistent kernel, one CTA per SM.  The work is a list of tiles, one per
// (layer l, request b, value head h) = one 128 x 128 fp32 state slab, ordered
// (l, b, key head, head in group); every CTA takes a contiguous range, so
// consecutive tiles usually share their key head and the q/k prologue
// (conv + SiLU + L2 of q and k, the Gram entries) is computed once per key
// head per CTA.
//
// Per tile:
//   * the state slab S0 arrives by TMA (four 32-column boxes, 128-byte
//     swizzle) into one of two stages, one tile ahead of use;
//   * the 128 row threads split S0 into tf32 hi + lo parts and store them in
//     tensor memory (operand A, lane = state row);
//   * one thread issues S0 [k_0..k_{N-1} | q_0..q_{N-1}] as three tf32 MMAs
//     per K step (hi*hi + hi*lo + lo*hi: products accurate to ~2^-20) into a
//     TMEM accumulator; [K|Q] hi/lo live in shared memory in the canonical
//     K-major 128-byte-swizzled layout (operand B);
//   * thread = state row: read its accumulator row, run the factored delta
//     recurrence over the nodes (delta_n = b_n (v_n - a_n S_p k_n) with
//     S_p k_n = gamma_p S0 k_n + sum_j g(j->p) delta_j k_j.k_n), write o_n,
//     and overwrite its S0 row in shared memory with the accepted state
//     gamma_acc S0 + sum_j g(j->acc) delta_j k_j^T;
//   * the slab goes back to global memory in place by TMA store.
// The conv window of the slot is persisted as in the CUDA-core kernel: each
// tile writes its value-head channels, and the last tile of a key head group
// to finish (arrival counter) writes the q/k channels.
#pragma once

#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_step.cuh"
#include "tc_ptx.cuh"

namespace lbx {

constexpr int kTcD = 128;             // head dimension of this kernel
constexpr int kTcRowThreads = 256;    // 8 warps: two per TMEM lane quadrant
constexpr int kTcThreads = kTcRowThreads + 32;  // + one control warp (TMA, MMA, TMEM)
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcAHi = 0, kTcALo = 128, kTcD0 = 256;  // TMEM column map
constexpr uint32_t kStageBytes = kTcD * kTcD * 4;    // one state slab, 64 KB

// Shared-memory layout for node capacity NMAX (k rows at [0, NMAX), q rows
// at [NMAX, 2*NMAX) of operand B / accumulator columns).
template <int NMAX>
struct TcLayout {
  static constexpr int NC = 2 * NMAX;
  static constexpr int kB = NC * kTcD * 4;          // one of B hi / B lo
  static constexpr int kNPair = NMAX * (NMAX - 1) / 2 + 1;
  static constexpr int TP = (NMAX + 3) & ~3;        // row pitch of T and W
  static constexpr int stage0 = 0;
  static constexpr int stage1 = stage0 + (int)kStageBytes;
  static constexpr int bhi = stage1 + (int)kStageBytes;
  static constexpr int blo = bhi + kB;
  static constexpr int v = blo + kB;                  // [NMAX][128] fp32 v_n of the tile's head
  static constexpr int del = v + NMAX * kTcD * 4;     // [NMAX][128] fp32 delta_n
  static constexpr int tm = del + NMAX * kTcD * 4;    // [NMAX][TP] T = (I + diag(b a) M)^-1
  static constexpr int wm = tm + NMAX * TP * 4;       // [NMAX][TP] W = Q T
  static constexpr int pj = wm + NMAX * TP * 4;       // int   [kNPair] parent-path nodes
  static constexpr int gkk = pj + 4 * kNPair;         // float [kNPair] k_j . k_n
  static constexpr int gkq = gkk + 4 * kNPair;        // float [kNPair] k_j . q_n
  static constexpr int ckk = gkq + 4 * kNPair;        // float [kNPair] g(j->p) k_j . k_n (per tile)
  static constexpr int ckq = ckk + 4 * kNPair;        // float [kNPair] g(j->p) k_j . q_n (per tile)
  static constexpr int tg_ = ckq + 4 * kNPair;        // float [NMAX] accepted-path coefficients
  static constexpr int tj = tg_ + 4 * NMAX;           // int   [NMAX] accepted-path nodes
  static constexpr int par = tj + 4 * NMAX;
  static constexpr int dep = par + 4 * NMAX;
  static constexpr int off = dep + 4 * NMAX;          // [NMAX + 1]
  static constexpr int win = off + 4 * (NMAX + 4);    // [NMAX][4]
  static constexpr int an = win + 16 * NMAX;
  static constexpr int bn = an + 4 * NMAX;
  static constexpr int gam = bn + 4 * NMAX;
  static constexpr int kqn = gam + 4 * NMAX;
  static constexpr int crow = kqn + 4 * NMAX;         // [4] conv-window sources (row threads)
  static constexpr int ccrow = crow + 16;             // [4] same, control warp's copy
  static constexpr int misc = ccrow + 16;             // ints: see kernel
  static constexpr int bars = (misc + 64 + 7) & ~7;   // 3 x uint64
  static constexpr int total = bars + 3 * 8;
  static_assert(kB % 1024 == 0, "operand B must keep 1024-byte alignment");
};

struct TcArgs {
  StepArgs s;
  int n_tiles;  // L * Bq * Hv
};

// Byte offset of element (row, k) inside a K-major, 128-byte-swizzled operand
// with `rows` rows and 128 fp32 columns: four 32-column atoms, each
// rows x 128 bytes; 16-byte chunk index XOR (row & 7).
__device__ __forceinline__ uint32_t sw128_off(int rows, int row, int k) {
  const int atom = k >> 5, chunk = (k >> 2) & 7;
  return (uint32_t)(atom * rows * 128 + row * 128 + ((chunk ^ (row & 7)) << 4) + ((k & 3) << 2));
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

// Conv-window persist of NCH channels (chan[i]) by one thread: every old
// entry and new x value is loaded before anything is written, so the loads
// of all channels overlap.  src[rr] >= 0: x row; < 0: old cache row -1-src.
template <int NCH>
__device__ __forceinline__ void persist_conv_batch(const int (&chan)[NCH], int K, int C,
                                                   const int (&src)[LBX_MAX_CONV_WIDTH - 1],
                                                   const uint16_t *x_lb, const float *cache_in,
                                                   float *cache_out) {
  float val[NCH][LBX_MAX_CONV_WIDTH - 1];
#pragma unroll
  for (int i = 0; i < NCH; ++i)
#pragma unroll
    for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr)
      if (rr < K - 1) {
        const int w = src[rr];
        val[i][rr] = w >= 0 ? bf2f(x_lb[(size_t)w * C + chan[i]])
                            : cache_in[(size_t)(-1 - w) * C + chan[i]];
      }
#pragma unroll
  for (int i = 0; i < NCH; ++i)
#pragma unroll
    for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr)
      if (rr < K - 1) cache_out[(size_t)rr * C + chan[i]] = val[i][rr];
}

template <int NMAX>
__global__ void __launch_bounds__(kTcThreads, 1)
    gdn_step_tc_kernel(const __grid_constant__ CUtensorMap tmap_state, const TcArgs T) {
  using Ly = TcLayout<NMAX>;
  constexpr int NC = Ly::NC;
  constexpr int TP = Ly::TP;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *stage[2] = {smem + Ly::stage0, smem + Ly::stage1};
  unsigned char *Bhi = smem + Ly::bhi;
  unsigned char *Blo = smem + Ly::blo;
  float *V = reinterpret_cast<float *>(smem + Ly::v);
  float *DEL = reinterpret_cast<float *>(smem + Ly::del);
  float *Tm = reinterpret_cast<float *>(smem + Ly::tm);
  float *Wm = reinterpret_cast<float *>(smem + Ly::wm);
  int *pj = reinterpret_cast<int *>(smem + Ly::pj);
  float *gkk = reinterpret_cast<float *>(smem + Ly::gkk);
  float *gkq = reinterpret_cast<float *>(smem + Ly::gkq);
  float *ckk = reinterpret_cast<float *>(smem + Ly::ckk);
  float *ckq = reinterpret_cast<float *>(smem + Ly::ckq);
  float *tg = reinterpret_cast<float *>(smem + Ly::tg_);
  int *tj = reinterpret_cast<int *>(smem + Ly::tj);
  int *par = reinterpret_cast<int *>(smem + Ly::par);
  int *dep = reinterpret_cast<int *>(smem + Ly::dep);
  int *off = reinterpret_cast<int *>(smem + Ly::off);
  int *win = reinterpret_cast<int *>(smem + Ly::win);
  float *an = reinterpret_cast<float *>(smem + Ly::an);
  float *bn = reinterpret_cast<float *>(smem + Ly::bn);
  float *gam = reinterpret_cast<float *>(smem + Ly::gam);
  float *kqn = reinterpret_cast<float *>(smem + Ly::kqn);
  int *crow = reinterpret_cast<int *>(smem + Ly::crow);
  int *ccrow = reinterpret_cast<int *>(smem + Ly::ccrow);
  int *misc = reinterpret_cast<int *>(smem + Ly::misc);
  // misc[0] error flag, [1] abort, [3] TMEM base, [4] accepted-path length
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + Ly::bars);  // [2]
  uint64_t *mma_bar = full_bar + 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool is_ctrl = warp == kTcRowThreads / 32;
  const int N = A.N, K = A.K, Hk = A.Hk, Hv = A.Hv, Bq = A.Bq;
  const int G = Hv / Hk;
  const int C = (2 * Hk + Hv) * kTcD;

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
  if (is_ctrl) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t *>(&misc[3]), kTcTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[3]);

  // tile -> state row of its slab
  auto tile_row = [&](int t) -> int {
    const int hg = t % G, rest = t / G;
    const int kh = rest % Hk, lb = rest / Hk;
    const int bq = lb % Bq, l = lb / Bq;
    const int h = kh * G + hg;
    return ((l * A.n_slots + A.slot[bq]) * Hv + h) * kTcD;
  };

  // control thread: prefetch the first tile
  const bool ctrl_lane = is_ctrl && lane == 0;
  int pending = -1;          // stage with an issued, not yet consumed load (control thread)
  uint32_t pending_par = 0;  // its phase parity
  if (ctrl_lane && count > 0) {
    const int row = tile_row(t_begin);
    ptx::mbar_arrive_expect_tx(&full_bar[0], kStageBytes);
    for (int a = 0; a < 4; ++a)
      ptx::tma_load_2d(stage[0] + a * (kStageBytes / 4), &tmap_state, a * 32, row, &full_bar[0]);
    pending = 0;
  }

  // row-thread identity: row r (TMEM lane), half hf (column half)
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int hf = (warp >> 2) & 1;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);  // this warp's lane quadrant

  // gates of the next tile, prefetched by threads tid < N
  float ga = 0.f, gb = 0.f;
  if (!is_ctrl && tid < N && count > 0) {
    const int t = t_begin, hg = t % G, rest = t / G, kh = rest % Hk, lbi = rest / Hk;
    ga = bf2f(A.a[((size_t)lbi * N + tid) * Hv + kh * G + hg]);
    gb = bf2f(A.b[((size_t)lbi * N + tid) * Hv + kh * G + hg]);
  }

  // control warp: the previous tile's value-head window persist is deferred
  // until the next tile's MMAs are running
  const uint16_t *pv_x = nullptr;
  const float *pv_in = nullptr;
  float *pv_out = nullptr;
  int pv_c0 = 0;
  int pv_src[LBX_MAX_CONV_WIDTH - 1] = {0, 0, 0};

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
    const uint16_t *x_lb = A.x + lb * N * C;
    const uint16_t *w_l = A.conv_w + (size_t)l * C * K;
    const float *cache_s = A.conv_cache + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
    float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
    const int32_t *par_b = A.parent + (size_t)bq * N;
    const int acc = A.accepted[bq];
    unsigned char *st = stage[s];

    if (!is_ctrl) {
      // ================= group prologue (new key head) =================
      if (rest != cur_group) {
        cur_group = rest;
        for (int i = tid; i < N; i += kTcRowThreads) {
          int dpt = 0;
          for (int m = i; m > 0; m = par_b[m]) ++dpt;
          par[i] = par_b[i];
          dep[i] = dpt;
          int m = i, past = 0;
          for (int j = 0; j < K; ++j) {
            if (m >= 0) {
              win[i * 4 + j] = m;
              m = par_b[m];
            } else {
              ++past;
              win[i * 4 + j] = -1 - (K - 1 - past);
            }
          }
        }
        if (tid == 32) window_sources(crow, K, acc, par_b);
        ptx::named_sync(1, kTcRowThreads);
        if (tid == 0) {
          off[0] = 0;
          for (int i = 0; i < N; ++i) off[i + 1] = off[i] + dep[i];
        }
        ptx::named_sync(1, kTcRowThreads);
        for (int i = tid; i < N; i += kTcRowThreads) {
          int j = par[i];
          for (int e = off[i]; e < off[i + 1]; ++e) {
            pj[e] = j;
            j = par[j];
          }
        }
        // q/k conv + SiLU + L2 -> operand B rows (hi / lo parts); q scaled.
        // All of a thread's units are loaded before any is reduced.
        {
          constexpr int GQ = kTcD / 8;  // 16 threads per (node, q|k)
          constexpr int U = (2 * NMAX * GQ + kTcRowThreads - 1) / kTcRowThreads;
          const int units = 2 * N * GQ;
          float v8[U][8], ss[U];
#pragma unroll
          for (int p = 0; p < U; ++p) {
            const int u = p * kTcRowThreads + tid;
            const int grp = u / GQ, li = u % GQ;
            const bool is_q = grp >= N;
            const int i = is_q ? grp - N : grp;
            if (u < units) {
              conv8(v8[p], win + i * 4, K, x_lb, C, w_l, cache_s,
                    (is_q ? 0 : Hk * kTcD) + kh * kTcD + li * 8);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[p][e] = 0.f;
            }
            ss[p] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss[p] = fmaf(v8[p][e], v8[p][e], ss[p]);
          }
#pragma unroll
          for (int p = 0; p < U; ++p)
#pragma unroll
            for (int o = GQ / 2; o > 0; o >>= 1) ss[p] += __shfl_xor_sync(0xffffffffu, ss[p], o);
#pragma unroll
          for (int p = 0; p < U; ++p) {
            const int u = p * kTcRowThreads + tid;
            if (u < units) {
              const int grp = u / GQ, li = u % GQ;
              const bool is_q = grp >= N;
              const int i = is_q ? grp - N : grp;
              const float scale = rsqrtf(ss[p] + A.l2_eps) * (is_q ? A.q_scale : 1.f);
              const int brow = is_q ? NMAX + i : i;
#pragma unroll
              for (int hq = 0; hq < 2; ++hq) {
                float4 hi, lo;
                float *ph = &hi.x, *pl = &lo.x;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float v = scale * v8[p][4 * hq + e];
                  const float vh = __uint_as_float(__float_as_uint(v) & 0xffffe000u);
                  ph[e] = vh;
                  pl[e] = v - vh;
                }
                const uint32_t o = sw128_off(NC, brow, li * 8 + 4 * hq);
                *reinterpret_cast<float4 *>(Bhi + o) = hi;
                *reinterpret_cast<float4 *>(Blo + o) = lo;
              }
            }
          }
          // zero the unused rows of operand B
          const int pad_rows = 2 * (NMAX - N);
          for (int idx = tid; idx < pad_rows * 32; idx += kTcRowThreads) {
            const int pr = idx / 32, q = idx % 32;
            const int brow = pr < NMAX - N ? N + pr : NMAX + N + (pr - (NMAX - N));
            const uint32_t o = sw128_off(NC, brow, 4 * q);
            *reinterpret_cast<float4 *>(Bhi + o) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(Blo + o) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        ptx::fence_proxy_async();
        ptx::named_sync(1, kTcRowThreads);
        // Gram entries: 8 threads per item; items are the parent-path pairs
        // (k_j.k_n, k_j.q_n for j = pj[e]) followed by the N diagonals k_n.q_n
        {
          const int npair = off[N];
          const int items = npair + N;
          const int sub = tid & 7;
          for (int base = 0; base < items; base += kTcRowThreads / 8) {
            const int item = base + (tid >> 3);
            const bool act = item < items;
            int j, n;
            if (!act) {
              j = 0, n = 0;
            } else if (item < npair) {
              j = pj[item];
              n = 0;
              while (off[n + 1] <= item) ++n;
            } else {
              j = item - npair, n = j;
            }
            float s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int k = 4 * (sub + 8 * c);
              const uint32_t oj = sw128_off(NC, j, k), on = sw128_off(NC, n, k),
                             oq = sw128_off(NC, NMAX + n, k);
              float4 kj = *reinterpret_cast<const float4 *>(Bhi + oj);
              float4 t4 = *reinterpret_cast<const float4 *>(Blo + oj);
              kj.x += t4.x, kj.y += t4.y, kj.z += t4.z, kj.w += t4.w;
              float4 kn = *reinterpret_cast<const float4 *>(Bhi + on);
              t4 = *reinterpret_cast<const float4 *>(Blo + on);
              kn.x += t4.x, kn.y += t4.y, kn.z += t4.z, kn.w += t4.w;
              float4 qn = *reinterpret_cast<const float4 *>(Bhi + oq);
              t4 = *reinterpret_cast<const float4 *>(Blo + oq);
              qn.x += t4.x, qn.y += t4.y, qn.z += t4.z, qn.w += t4.w;
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
        ptx::named_sync(1, kTcRowThreads);
      }

      // ================= per-tile preparation =================
      if (tid < N) {
        an[tid] = ga;
        bn[tid] = gb;
      }
      ptx::named_sync(1, kTcRowThreads);
      // per parent-path pair: g(j->p) times the Gram entries; gamma_p per node
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
      // ================= S0 -> tensor memory (tf32 hi / lo) =================
      if (!ptx::mbar_wait(&full_bar[s], (uint32_t)((it >> 1) & 1))) {
        if (A.status) *A.status = LBX_ETIMEOUT;
        atomicExch(&misc[1], 1);
      }
      {
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
          uint32_t vh[32], vl[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int k = hf * 64 + c32 * 32 + 4 * q;
            const float4 x4 = *reinterpret_cast<const float4 *>(st + sw128_off(kTcD, r, k));
            const float *px = &x4.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t hb = __float_as_uint(px[e]) & 0xffffe000u;
              vh[4 * q + e] = hb;
              vl[4 * q + e] = __float_as_uint(px[e] - __uint_as_float(hb));
            }
          }
          const uint32_t col = (uint32_t)(hf * 64 + c32 * 32);
          ptx::tmem_st32(tq + kTcAHi + col, vh);
          ptx::tmem_st32(tq + kTcALo + col, vl);
        }
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
    }
    __syncthreads();  // ---------------------------------------------- S1
    if (misc[1]) break;

    if (is_ctrl) {
      if (lane == 0) {
        // the MMAs: D = S0 [K|Q]^T, three tf32 passes over K = 128
        ptx::tc_fence_after();
        constexpr uint32_t idesc = ptx::idesc_tf32(128, NC);
        const uint32_t bhi_a = ptx::smem_u32(Bhi), blo_a = ptx::smem_u32(Blo);
        uint32_t accum = 0;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t a_col = pass == 2 ? kTcALo : kTcAHi;
          const uint32_t b_base = pass == 1 ? blo_a : bhi_a;
#pragma unroll
          for (int ks = 0; ks < kTcD / 8; ++ks) {
            const uint32_t baddr = b_base + (uint32_t)((ks >> 2) * (NC * 128) + (ks & 3) * 32);
            ptx::mma_tf32_ts(tmem + kTcD0, tmem + a_col + 8 * ks, ptx::sdesc_sw128(baddr), idesc,
                             accum);
            accum = 1;
          }
        }
        ptx::mma_commit(mma_bar);
        // prefetch the next tile into the other stage once its previous
        // contents (tile it-1) have been read by their TMA store
        if (it + 1 < count) {
          const int s2 = (it + 1) & 1;
          ptx::bulk_wait_read_all();
          const int row = tile_row(t + 1);
          ptx::mbar_arrive_expect_tx(&full_bar[s2], kStageBytes);
          for (int a = 0; a < 4; ++a)
            ptx::tma_load_2d(stage[s2] + a * (kStageBytes / 4), &tmap_state, a * 32, row,
                             &full_bar[s2]);
          pending = s2;
          pending_par = (uint32_t)(((it + 1) >> 1) & 1);
        } else {
          pending = -1;
        }
        // conv-window sources for this tile's persist work
        window_sources(ccrow, K, acc, par_b);
      }
      // value-head window of the previous tile (its v conv finished before
      // that tile's S3)
      if (pv_x != nullptr) {
        int ch[kTcD / 32];
#pragma unroll
        for (int i = 0; i < kTcD / 32; ++i) ch[i] = pv_c0 + lane + 32 * i;
        persist_conv_batch(ch, K, C, pv_src, pv_x, pv_in, pv_out);
      }
      __syncwarp();
      int src[LBX_MAX_CONV_WIDTH - 1];
#pragma unroll
      for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr) src[rr] = rr < K - 1 ? ccrow[rr] : 0;
      // arrival: this CTA has finished reading the old q/k window of the
      // key head (group prologue, before S1); the last of the G tiles of
      // the group writes the new q/k window
      int last = 0;
      if (lane == 0) {
        __threadfence();
        unsigned int *cnt = A.counters + lb * Hk + kh;
        const unsigned int prev = atomicAdd(cnt, 1u);
        last = prev == (unsigned int)(G - 1);
        if (last) {
          atomicExch(cnt, 0u);
          __threadfence();
        }
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        int ch[2 * kTcD / 32];
#pragma unroll
        for (int i = 0; i < 2 * kTcD / 32; ++i) {
          const int j = lane + 32 * i;
          ch[i] = j < kTcD ? kh * kTcD + j : Hk * kTcD + kh * kTcD + (j - kTcD);
        }
        persist_conv_batch(ch, K, C, src, x_lb, cache_s, cache_o);
      }
      pv_x = x_lb, pv_in = cache_s, pv_out = cache_o, pv_c0 = 2 * Hk * kTcD + h * kTcD;
#pragma unroll
      for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr) pv_src[rr] = src[rr];
    } else {
      // ======== while the MMAs run: warp 0 builds T and W, the rest v ========
      if (warp == 0) {
        // T = (I + diag(b a) M)^-1, one column per lane, rows in node order;
        // M[n][j] = g(j->p) k_j.k_n on the parent path of n.
        const int m = lane;
        for (int n = 0; n < N; ++n) {
          const float d_n = bn[n] * an[n];
          float tv = (m == n) ? 1.f : 0.f;
          for (int e = off[n]; e < off[n + 1]; ++e) {
            const float tjm = m < TP ? Tm[pj[e] * TP + m] : 0.f;
            tv = fmaf(-d_n * ckk[e], tjm, tv);
          }
          if (m < TP) Tm[n * TP + m] = tv;
          __syncwarp();
        }
        if (lane == 0) {
          // accepted path: acc itself, then its parent path (coefficient g * a_acc)
          int cnt = 0;
          tj[cnt] = acc;
          tg[cnt] = 1.f;
          ++cnt;
          int j = par[acc];
          float g = an[acc];
          for (int e = off[acc]; e < off[acc + 1]; ++e) {
            tj[cnt] = pj[e];
            tg[cnt] = g;
            ++cnt;
            g *= an[j];
            j = par[j];
          }
          misc[4] = cnt;
        }
      } else {
        // v of head h for all 128 rows (conv + SiLU), V[node][row]
        constexpr int GV = kTcD / 8;
        constexpr int NT = kTcRowThreads - 32;
        constexpr int U = (NMAX * GV + NT - 1) / NT;
        const int units = N * GV;
        const int vt = tid - 32;
#pragma unroll
        for (int p = 0; p < U; ++p) {
          const int u = p * NT + vt;
          if (u < units) {
            const int i = u / GV, li = u % GV;
            float v8[8];
            conv8(v8, win + i * 4, K, x_lb, C, w_l, cache_s, 2 * Hk * kTcD + h * kTcD + li * 8);
            float4 *dst = reinterpret_cast<float4 *>(V + i * kTcD + li * 8);
            dst[0] = make_float4(v8[0], v8[1], v8[2], v8[3]);
            dst[1] = make_float4(v8[4], v8[5], v8[6], v8[7]);
          }
        }
      }
      ptx::named_sync(1, kTcRowThreads);
      // W = Q T, rows in parallel (warp per node): Q[n][j] = a_n g(j->p)
      // k_j.q_n on the parent path, Q[n][n] = k_n.q_n
      for (int n = warp; n < N; n += kTcRowThreads / 32) {
        if (lane < TP) {
          const float a_n = an[n];
          float wv = kqn[n] * Tm[n * TP + lane];
          for (int e = off[n]; e < off[n + 1]; ++e)
            wv = fmaf(a_n * ckq[e], Tm[pj[e] * TP + lane], wv);
          Wm[n * TP + lane] = wv;
        }
      }
      ptx::named_sync(1, kTcRowThreads);

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

      // rhs_n = b_n v_n - b_n a_n gamma_p S0 k_n ; delta = T rhs
      float rhs[NMAX];
#pragma unroll
      for (int n = 0; n < NMAX; ++n)
        rhs[n] = n < N ? bn[n] * fmaf(-an[n] * gam[n], dv[n], V[n * kTcD + r]) : 0.f;
      if (hf == 0) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
          if (n < N) {
            float d = 0.f;
#pragma unroll
            for (int m4 = 0; m4 <= n / 4; ++m4) {
              const float4 t4 = *reinterpret_cast<const float4 *>(Tm + n * TP + 4 * m4);
              d = fmaf(t4.x, rhs[4 * m4], d);
              if (4 * m4 + 1 <= n) d = fmaf(t4.y, rhs[4 * m4 + 1], d);
              if (4 * m4 + 2 <= n) d = fmaf(t4.z, rhs[4 * m4 + 2], d);
              if (4 * m4 + 3 <= n) d = fmaf(t4.w, rhs[4 * m4 + 3], d);
            }
            DEL[n * kTcD + r] = d;
          }
        }
      } else {
        // o_n = a_n gamma_p S0 q_n + (W rhs)_n
        float *o_base = A.o + (lb * N) * (size_t)Hv * kTcD + (size_t)h * kTcD + r;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
          if (n < N) {
            float ov = an[n] * gam[n] * dv[NMAX + n];
#pragma unroll
            for (int m4 = 0; m4 <= n / 4; ++m4) {
              const float4 w4 = *reinterpret_cast<const float4 *>(Wm + n * TP + 4 * m4);
              ov = fmaf(w4.x, rhs[4 * m4], ov);
              if (4 * m4 + 1 <= n) ov = fmaf(w4.y, rhs[4 * m4 + 1], ov);
              if (4 * m4 + 2 <= n) ov = fmaf(w4.z, rhs[4 * m4 + 2], ov);
              if (4 * m4 + 3 <= n) ov = fmaf(w4.w, rhs[4 * m4 + 3], ov);
            }
            __stcs(o_base + (size_t)n * Hv * kTcD, ov);
          }
        }
      }
      ptx::named_sync(1, kTcRowThreads);

      // ================= accepted state rows, in place =================
      {
        const int ntgt = misc[4];
        const float gacc = gam[acc] * an[acc];
        float4 accv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)
          accv[q] = f4_scale(gacc, *reinterpret_cast<const float4 *>(
                                       st + sw128_off(kTcD, r, hf * 64 + 4 * q)));
        for (int m = 0; m < ntgt; ++m) {
          const int j = tj[m];
          const float coef = tg[m] * DEL[j * kTcD + r];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const uint32_t ok = sw128_off(NC, j, hf * 64 + 4 * q);
            float4 kj = *reinterpret_cast<const float4 *>(Bhi + ok);
            const float4 kl = *reinterpret_cast<const float4 *>(Blo + ok);
            kj.x += kl.x, kj.y += kl.y, kj.z += kl.z, kj.w += kl.w;
            f4_fma(accv[q], coef, kj);
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q)
          *reinterpret_cast<float4 *>(st + sw128_off(kTcD, r, hf * 64 + 4 * q)) = accv[q];
      }
      // gates of the next tile
      if (tid < N && it + 1 < count) {
        const int t2 = t + 1, hg2 = t2 % G, rest2 = t2 / G, kh2 = rest2 % Hk, lb2 = rest2 / Hk;
        ga = bf2f(A.a[((size_t)lb2 * N + tid) * Hv + kh2 * G + hg2]);
        gb = bf2f(A.b[((size_t)lb2 * N + tid) * Hv + kh2 * G + hg2]);
      }
      ptx::fence_proxy_async();
      ptx::tc_fence_before();
    }
    __syncthreads();  // ---------------------------------------------- S3
    if (misc[1]) break;
    if (is_ctrl) {
      if (lane == 0) {
        const int row = tile_row(t);
        for (int a = 0; a < 4; ++a)
          ptx::tma_store_2d(&tmap_state, a * 32, row, st + a * (kStageBytes / 4));
        ptx::bulk_commit();
      }
    }
  }
  // value-head window of the last tile
  if (is_ctrl && pv_x != nullptr && !misc[1]) {
    int ch[kTcD / 32];
#pragma unroll
    for (int i = 0; i < kTcD / 32; ++i) ch[i] = pv_c0 + lane + 32 * i;
    persist_conv_batch(ch, K, C, pv_src, pv_x, pv_in, pv_out);
  }

  // ---- drain: outstanding loads (only after an abort) and stores ----
  if (ctrl_lane) {
    if (pending >= 0 && misc[1]) (void)ptx::mbar_wait(&full_bar[pending], pending_par);
    ptx::bulk_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (is_ctrl) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace lbx
