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
  static constexpr int stage0 = 0;
  static constexpr int stage1 = stage0 + (int)kStageBytes;
  static constexpr int bhi = stage1 + (int)kStageBytes;
  static constexpr int blo = bhi + kB;
  static constexpr int v = blo + kB;                  // [NMAX][128] fp32
  static constexpr int del = v + NMAX * kTcD * 4;     // [NMAX][128] fp32
  static constexpr int pj = del + NMAX * kTcD * 4;    // int   [kNPair]
  static constexpr int gkk = pj + 4 * kNPair;         // float [kNPair]
  static constexpr int gkq = gkk + 4 * kNPair;
  static constexpr int ckk = gkq + 4 * kNPair;
  static constexpr int ckq = ckk + 4 * kNPair;
  static constexpr int tg_ = ckq + 4 * kNPair;        // float [NMAX] target coefficients
  static constexpr int tj = tg_ + 4 * NMAX;           // int   [NMAX] target nodes
  static constexpr int par = tj + 4 * NMAX;
  static constexpr int dep = par + 4 * NMAX;
  static constexpr int off = dep + 4 * NMAX;          // [NMAX + 1]
  static constexpr int win = off + 4 * (NMAX + 4);    // [NMAX][4]
  static constexpr int an = win + 16 * NMAX;
  static constexpr int bn = an + 4 * NMAX;
  static constexpr int gam = bn + 4 * NMAX;
  static constexpr int kqn = gam + 4 * NMAX;
  static constexpr int crow = kqn + 4 * NMAX;         // [4]
  static constexpr int misc = crow + 16;              // ints: see kernel
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

template <int NMAX>
__global__ void __launch_bounds__(kTcThreads, 1)
    gdn_step_tc_kernel(const __grid_constant__ CUtensorMap tmap_state, const TcArgs T) {
  using Ly = TcLayout<NMAX>;
  constexpr int NC = Ly::NC;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *stage[2] = {smem + Ly::stage0, smem + Ly::stage1};
  unsigned char *Bhi = smem + Ly::bhi;
  unsigned char *Blo = smem + Ly::blo;
  float *V = reinterpret_cast<float *>(smem + Ly::v);
  float *DEL = reinterpret_cast<float *>(smem + Ly::del);
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
  int *misc = reinterpret_cast<int *>(smem + Ly::misc);
  // misc[0] error flag, [1] abort, [2] last arriver, [3] TMEM base, [4] ntgt
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

  // tile -> (l, b, kh, hg) and the state row of its slab
  auto tile_row = [&](int t) -> int {
    const int hg = t % G, rest = t / G;
    const int kh = rest % Hk, lb = rest / Hk;
    const int bq = lb % Bq, l = lb / Bq;
    const int h = kh * G + hg;
    return ((l * A.n_slots + A.slot[bq]) * Hv + h) * kTcD;
  };

  // control thread: prefetch the first tile
  const bool ctrl_lane = is_ctrl && lane == 0;
  int pending = -1;         // stage with an issued, not yet consumed load (control thread)
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
    const int32_t *par_b = A.parent + (size_t)bq * N;
    const int acc = A.accepted[bq];
    unsigned char *st = stage[s];

    if (!is_ctrl) {
      // ================= group prologue (new key head) =================
      if (rest != cur_group) {
        cur_group = rest;
        for (int i = tid; i < N; i += kTcRowThreads) {
          const int p = par_b[i];
          int dpt = 0;
          for (int m = i; m > 0; m = par_b[m]) ++dpt;
          par[i] = p;
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
        if (tid == 0) {
          // new conv-window sources: row rr <- (K-2-rr)-th ancestor of acc,
          // or old cache row depth(acc)+1+rr when the path is too short
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
            crow[rr] = w;
          }
        }
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
        // q/k conv + SiLU + L2 -> operand B rows (hi / lo parts); q scaled
        {
          constexpr int GQ = kTcD / 8;  // 16 threads per (node, q|k)
          const int units = 2 * N * GQ;
          for (int base = 0; base < units; base += kTcRowThreads) {
            const int u = base + tid;
            const bool act = u < units;
            const int grp = act ? u / GQ : 0, li = u % GQ;
            const bool is_q = grp >= N;
            const int i = is_q ? grp - N : grp;
            const int c0 = (is_q ? 0 : Hk * kTcD) + kh * kTcD + li * 8;
            float v8[8];
            if (act) {
              conv8(v8, win + i * 4, K, x_lb, C, w_l, cache_s, c0);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[e] = 0.f;
            }
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(v8[e], v8[e], ss);
#pragma unroll
            for (int o = GQ / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float scale = rsqrtf(ss + A.l2_eps) * (is_q ? A.q_scale : 1.f);
            if (act) {
              const int brow = is_q ? NMAX + i : i;
#pragma unroll
              for (int hq = 0; hq < 2; ++hq) {
                float4 hi, lo;
                float *ph = &hi.x, *pl = &lo.x;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float v = scale * v8[4 * hq + e];
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
        // Gram entries (warp per node): k_j.k_i and k_j.q_i for j on the
        // parent path of i, and k_i.q_i
        for (int i = warp; i < N; i += kTcRowThreads / 32) {
          const uint32_t oki = sw128_off(NC, i, 4 * lane), oqi = sw128_off(NC, NMAX + i, 4 * lane);
          float4 ki = *reinterpret_cast<const float4 *>(Bhi + oki);
          float4 t4 = *reinterpret_cast<const float4 *>(Blo + oki);
          ki.x += t4.x, ki.y += t4.y, ki.z += t4.z, ki.w += t4.w;
          float4 qi = *reinterpret_cast<const float4 *>(Bhi + oqi);
          t4 = *reinterpret_cast<const float4 *>(Blo + oqi);
          qi.x += t4.x, qi.y += t4.y, qi.z += t4.z, qi.w += t4.w;
          const float kq = warp_sum(dot4(ki, qi));
          if (lane == 0) kqn[i] = kq;
          for (int e = off[i]; e < off[i + 1]; ++e) {
            const uint32_t okj = sw128_off(NC, pj[e], 4 * lane);
            float4 kj = *reinterpret_cast<const float4 *>(Bhi + okj);
            t4 = *reinterpret_cast<const float4 *>(Blo + okj);
            kj.x += t4.x, kj.y += t4.y, kj.z += t4.z, kj.w += t4.w;
            const float s1 = warp_sum(dot4(kj, ki));
            const float s2 = warp_sum(dot4(kj, qi));
            if (lane == 0) {
              gkk[e] = s1;
              gkq[e] = s2;
            }
          }
        }
        ptx::named_sync(1, kTcRowThreads);
      }

      // ================= per-tile preparation =================
      for (int i = tid; i < N; i += kTcRowThreads) {
        an[i] = bf2f(A.a[(lb * N + i) * Hv + h]);
        bn[i] = bf2f(A.b[(lb * N + i) * Hv + h]);
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
      // v of head h for all 128 rows (conv + SiLU), V[node][row]
      {
        constexpr int GV = kTcD / 8;
        const int units = N * GV;
        for (int u = tid; u < units; u += kTcRowThreads) {
          const int i = u / GV, li = u % GV;
          const int c0 = 2 * Hk * kTcD + h * kTcD + li * 8;
          float v8[8];
          conv8(v8, win + i * 4, K, x_lb, C, w_l, cache_s, c0);
          float4 *dst = reinterpret_cast<float4 *>(V + i * kTcD + li * 8);
          dst[0] = make_float4(v8[0], v8[1], v8[2], v8[3]);
          dst[1] = make_float4(v8[4], v8[5], v8[6], v8[7]);
        }
      }
      ptx::named_sync(1, kTcRowThreads);
      if (tid == 0) {
        // accepted path: acc itself, then its parent path (coefficient g * a_acc)
        int m = 0;
        tj[m] = acc;
        tg[m] = 1.f;
        ++m;
        int j = par[acc];
        float g = an[acc];
        for (int e = off[acc]; e < off[acc + 1]; ++e) {
          tj[m] = pj[e];
          tg[m] = g;
          ++m;
          g *= an[j];
          j = par[j];
        }
        misc[4] = m;
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

      // ================= conv-window persist =================
      {
        float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
        if (tid < kTcD)
          persist_conv_channel(2 * Hk * kTcD + h * kTcD + tid, K, C, crow, x_lb, cache_s, cache_o);
        if (tid == 0) {
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
      }
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
      }
      __syncwarp();
    } else {
      // q/k conv-window channels, by the last tile of the key-head group
      if (misc[2]) {
        float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;
        const int j = tid;  // 256 threads = 2 * 128 channels
        persist_conv_channel(j < kTcD ? kh * kTcD + j : Hk * kTcD + kh * kTcD + (j - kTcD), K, C,
                             crow, x_lb, cache_s, cache_o);
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

      // ================= delta recurrence (one thread per row) =================
      if (hf == 0) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
          if (n < N) {
            float u = gam[n] * dv[n];
            for (int e = off[n]; e < off[n + 1]; ++e) u = fmaf(ckk[e], DEL[pj[e] * kTcD + r], u);
            DEL[n * kTcD + r] = bn[n] * (V[n * kTcD + r] - an[n] * u);
          }
        }
      }
      ptx::named_sync(1, kTcRowThreads);

      // ================= o_n = a_n (S_p q_n) + delta_n (k_n . q_n) =================
      {
        float *o_base = A.o + (lb * N) * (size_t)Hv * kTcD + (size_t)h * kTcD + r;
        auto emit = [&](int n, float sq) {
          float u = gam[n] * sq;
          for (int e = off[n]; e < off[n + 1]; ++e) u = fmaf(ckq[e], DEL[pj[e] * kTcD + r], u);
          const float ov = fmaf(an[n], u, kqn[n] * DEL[n * kTcD + r]);
          __stcs(o_base + (size_t)n * Hv * kTcD, ov);
        };
        if (hf == 0) {
#pragma unroll
          for (int n = 0; n < NMAX / 2; ++n)
            if (n < N) emit(n, dv[NMAX + n]);
        } else {
#pragma unroll
          for (int n = NMAX / 2; n < NMAX; ++n)
            if (n < N) emit(n, dv[NMAX + n]);
        }
      }

      // ================= accepted state rows, in place =================
      {
        const int ntgt = misc[4];
        const float gacc = gam[acc] * an[acc];
        for (int q = 0; q < 16; ++q) {
          const int k = hf * 64 + 4 * q;
          float4 *p = reinterpret_cast<float4 *>(st + sw128_off(kTcD, r, k));
          float4 accv = f4_scale(gacc, *p);
          for (int m = 0; m < ntgt; ++m) {
            const int j = tj[m];
            const float coef = tg[m] * DEL[j * kTcD + r];
            const uint32_t ok = sw128_off(NC, j, k);
            float4 kj = *reinterpret_cast<const float4 *>(Bhi + ok);
            const float4 kl = *reinterpret_cast<const float4 *>(Blo + ok);
            kj.x += kl.x, kj.y += kl.y, kj.z += kl.z, kj.w += kl.w;
            f4_fma(accv, coef, kj);
          }
          *p = accv;
        }
      }
      ptx::fence_proxy_async();
      ptx::tc_fence_before();
    }
    __syncthreads();  // ---------------------------------------------- S3
    if (misc[1]) break;
    if (ctrl_lane) {
      const int row = tile_row(t);
      for (int a = 0; a < 4; ++a)
        ptx::tma_store_2d(&tmap_state, a * 32, row, st + a * (kStageBytes / 4));
      ptx::bulk_commit();
    }
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
