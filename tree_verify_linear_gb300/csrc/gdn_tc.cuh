// gdn_tc.cuh -- fused tree-verify step on tensor cores (sm_103a, d = 128).
//
// Up to 24 nodes two CTAs share each SM (at most 113 KB of shared memory and
// 256 TMEM columns each), so the latency-bound phases of one CTA overlap the
// other's; a CTA has 8 warps, warps w and w + 4 share TMEM lane quadrant w,
// and each state row (= TMEM lane) has two threads, one per part: of the 128
// columns when the state is split and written back, of the nodes in the row
// work.  Larger capacities take one CTA of 16 warps per SM and four parts
// (warps w, w + 4, w + 8, w + 12 on quadrant w).
// The work is a list of tiles, one per (layer l, request b, value head h) =
// one 128 x 128 fp32 state slab, ordered (l, b, key head, head in group);
// every CTA takes a contiguous range, so consecutive tiles usually share
// their request and key head.  The prep kernel (gdn_tc_prep.cuh) has already
// built, per request, the tree tables and, per key head, the [K|Q] operand
// and the Gram entries; the step kernel bulk-copies them from the workspace
// when the request or the key head changes.
//
// Nodes are relabelled per request so that the accepted path comes first
// (root = 0, ..., accepted node = P-1) and the rest follow in index order;
// parents still precede children.  Thread 0 also issues the bulk-async copies
// of the state slab S0 (TMA, four 32-column boxes, 128-byte swizzle) into the
// stage, as soon as the previous tile's state store has read it (at two CTAs
// per SM the next tile's slab is first prefetched into L2 a tile ahead), and
// of the raw inputs, cached window rows and conv weights of the value head's
// 128 channels into the staging buffer, one tile ahead.  A tile computes its v
// conv first, while its slab and its value-head record are still on the way,
// and writes o while MMA3 runs.
//
// With the factored delta rule S_n = gamma_n S0 + sum_{j in path(n)}
// g(j->n) delta_j k_j^T (g = product of the gates strictly after j), every
// delta of a row follows from rhs_n = b_n v_n - b_n a_n gamma_p(n) S0 k_n as
// delta = T rhs, T = (I + diag(b a) M)^-1 with M[n][j] = g(j->p(n)) k_j.k_n
// on the parent path, and o = diag(a gamma) S0 q + W rhs with W = Q T,
// Q[n][j] = a_n g(j->p(n)) k_j.q_n, Q[n][n] = k_n.q_n.  Per tile, three
// tensor-core products (bf16 hi + lo operands, three passes hi*hi + hi*lo +
// lo*hi, relative error ~2^-17, fp32 accumulators in TMEM) do the row work:
//   MMA1  [S0 k_n | S0 q_n]      = S0 [K | Q]^T      (A = S0 in TMEM, K = 128)
//   MMA2  [delta_n | (W rhs)_n]  = rhs [T | W]^T     (A = rhs in TMEM, K = N)
//   MMA3  sum_j c_j delta_j k_j^T = (c . delta) K     (A = path deltas, K = P,
//         B = the K rows of the operand read N-major)
// and the accepted state gamma_acc S0 + MMA3 is formed in place over the
// staged S0 (exact fp32 S0, the MMA3 accumulator from tensor memory) and
// written back by TMA stores of the four boxes.  T and W (shared by the 128
// rows) are built by one lane per (node, ancestor-or-self) pair, each walking
// its stretch of the parent path, with no barriers.  Loops over nodes are unrolled to the node capacity NMAX
// and run without run-time guards: padding nodes carry zero gates, taps
// beyond the conv width zero weights, every load a clamped, valid index.
// The conv window of the slot is persisted in place: every value channel by
// its row thread here, the q/k channels by the prep kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "gdn_common.cuh"
#include "gdn_step.cuh"
#include "tc_ptx.cuh"

namespace lbx {

constexpr int kTcD = 128;                      // head dimension of this kernel
constexpr int kTcThreads = 256;                // 8 warps, two threads per state row
constexpr int kTcCtasPerSm = 2;
constexpr uint32_t kTcTmemCols = 256;          // per CTA: two CTAs fill the 512 columns
constexpr uint32_t kStageBytes = kTcD * kTcD * 4;  // one state slab, 64 KB
constexpr int kTcMaxSmem = 113 * 1024;             // two CTAs per SM

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Resources of the tree step by node capacity: up to 24 nodes two CTAs of 8
// warps share an SM (256 TMEM columns and at most 113 KB of shared memory
// each), with two threads per state row; larger capacities (up to 64) take
// one CTA of 16 warps per SM with all 512 TMEM columns, four threads per
// state row (parts: each has a quarter of the nodes and columns).  The
// prep kernel handles prep_heads value heads at a time (its per-head scratch
// grows with NMAX^2); at the large capacities two of its 16-warp CTAs share
// an SM (64 registers per thread, at most 113 KB of shared memory each).
template <int NMAX>
struct TcRes {
  static constexpr int ctas = NMAX <= 24 ? 2 : 1;
  static constexpr uint32_t tmem_cols = NMAX <= 24 ? 256u : 512u;
  static constexpr int max_smem = NMAX <= 24 ? 113 * 1024 : 227 * 1024;
  static constexpr int prep_ctas = NMAX <= 24 ? 4 : 2;
  static constexpr int prep_heads = NMAX <= 24 ? 4 : 3;
  static constexpr int prep_threads = NMAX <= 24 ? 256 : 512;
  static constexpr int parts = NMAX <= 24 ? 2 : 4;  // threads per state row
  static constexpr int threads = 128 * parts;
};

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

// Per-request tree tables in the new labels (built by the prep kernel, one
// bulk copy into the step kernel): parent-path nodes pj and their node pn per
// (node, strict ancestor) pair, node ln per (node, ancestor-or-self) lane and
// the byte offset lofs of the lane's T entry in the [T|W] operand, parents,
// depths, pair and lane offsets, conv window sources (input x row >= 0, or
// cached row -1-w), label maps, the nodes in conv order (those whose window
// lies inside the tree first), new-window sources and {P = accepted-path
// length, lanes, pairs, nodes whose window lies inside the tree}.
template <int NMAX>
struct TabLayout {
  static constexpr int kNPair = NMAX * (NMAX - 1) / 2 + 1;
  static constexpr int kNLane = NMAX * (NMAX + 1) / 2;
  static constexpr int pj = 0;                          // uint8 [kNPair]
  static constexpr int pn = pj + round_up(kNPair, 16);  // uint8 [kNPair]
  static constexpr int ln = pn + round_up(kNPair, 16);  // uint8 [kNLane]
  static constexpr int lofs = ln + round_up(kNLane, 16);  // uint16 [kNLane]
  static constexpr int par = lofs + round_up(2 * kNLane, 16);  // int [NMAX]
  static constexpr int dep = par + 4 * round_up(NMAX, 4);
  static constexpr int off = dep + 4 * round_up(NMAX, 4);      // [NMAX + 4]
  static constexpr int off2 = off + 4 * (NMAX + 4);            // [NMAX + 4]
  static constexpr int win = off2 + 4 * (NMAX + 4);            // [NMAX][4]
  static constexpr int n2o = win + 16 * NMAX;
  static constexpr int o2n = n2o + 4 * round_up(NMAX, 4);
  static constexpr int corder = o2n + 4 * round_up(NMAX, 4);  // [NMAX] conv order
  static constexpr int crow = corder + 4 * round_up(NMAX, 4);  // [4]
  static constexpr int meta = crow + 16;                       // [4] P, lanes, pairs
  static constexpr int bytes = meta + 16;
  static_assert(win % 16 == 0 && bytes % 16 == 0, "alignment");
};

// Gram entries of one key head (prep kernel only): k_j.k_n and k_j.q_n of
// the parent-path pairs, then the diagonals k_n.q_n.
template <int NMAX>
struct GramLayout {
  static constexpr int kNPairP = round_up(NMAX * (NMAX - 1) / 2 + 1, 4);
  static constexpr int gkk = 0;
  static constexpr int gkq = gkk + 4 * kNPairP;
  static constexpr int kqn = gkq + 4 * kNPairP;
  static constexpr int bytes = kqn + 4 * round_up(NMAX, 4);
  static_assert(bytes % 16 == 0, "alignment");
};

// Per-value-head record (built by the prep kernel, bulk-copied per tile): in
// the new labels the gates a, b, gamma of the parent (product of the
// ancestors' gates), the accepted-path coefficients g(j->acc), gamma of the
// accepted node, then the T and the W entries of the tree's (node,
// ancestor-or-self) lanes.  A record's slot holds every lane a tree of NMAX
// nodes can have; only used(lanes) bytes of it are written and read.
template <int NMAX>
struct HeadLayout {
  static constexpr int kNLaneP = round_up(NMAX * (NMAX + 1) / 2, 4);
  static constexpr int NP = round_up(NMAX, 4);
  static constexpr int an = 0;                 // float [NP]
  static constexpr int bn = an + 4 * NP;
  static constexpr int gam = bn + 4 * NP;
  static constexpr int cpa = gam + 4 * NP;
  static constexpr int gacc = cpa + 4 * NP;    // float [4]
  static constexpr int tw = gacc + 16;         // float [2][lanes4]: T, then W
  static constexpr int bytes = tw + 8 * kNLaneP;
  // lanes rounded up to 4: the W entries start that many floats after T's
  __host__ __device__ static constexpr int lanes4(int lanes) { return round_up(lanes, 4); }
  __host__ __device__ static constexpr int used(int lanes) { return tw + 8 * lanes4(lanes); }
  static_assert(tw % 16 == 0 && bytes % 16 == 0, "alignment");
};

template <int NMAX>
struct TcLayout {
  using CS = ConvStage<NMAX>;
  static constexpr int NC = 2 * NMAX;                 // rows of [K | Q] and of [T | W]
  static constexpr int R1 = 2 * NC;                   // [K|Q] hi rows, then [K|Q] lo rows
  static constexpr int KP = round_up(NMAX, 16);       // node dimension padded to the MMA K step
  static constexpr int kB = R1 * kTcD * 2;            // [K|Q] hi and lo (bf16, 128-byte swizzle)
  static constexpr int kB2 = NC * KP * 2;             // one of [T|W] hi / lo (bf16, no swizzle)
  static constexpr int TP = (NMAX + 3) & ~3;          // row pitch of the fp32 T scratch
  // TMEM columns: S0 hi | lo; the two halves of [S0 k | S0 q] (hi-row and
  // lo-row products); rhs or path deltas (hi | lo).  [delta | W rhs] reuses
  // the first half of the MMA1 accumulator, the MMA3 accumulator the S0
  // columns (free once MMA1 has completed).
  static constexpr uint32_t cA1 = 0, cD1 = 128, cA2 = cD1 + R1, cD2 = cD1;
  static_assert(cA2 + KP <= TcRes<NMAX>::tmem_cols, "tensor memory");
  // byte distance from a T entry of [T|W] to the W entry of the same lane
  static constexpr int kWOff = (NMAX / 8) * KP * 16;
  static_assert(NMAX % 8 == 0, "W rows start at an 8-row group");
  static constexpr int stage = 0;
  static constexpr int b1 = stage + (int)kStageBytes;  // [K|Q] image of the key head
  static constexpr int b2hi = b1 + kB;
  static constexpr int b2lo = b2hi + kB2;
  static constexpr int stg = round_up(b2lo + kB2, 128);  // value-head conv inputs
  static constexpr int tb = stg + CS::bytes;           // tree tables
  static constexpr int hr = tb + TabLayout<NMAX>::bytes;  // value-head record
  static constexpr int misc = hr + HeadLayout<NMAX>::bytes;  // ints, see kernel
  static constexpr int bars = (misc + 64 + 7) & ~7;   // 6 x uint64
  static constexpr int total = bars + 6 * 8;
  static constexpr int smem_bytes = total;
  static_assert(kB % 1024 == 0, "operand [K|Q] must keep 1024-byte alignment");
  static_assert(smem_bytes <= TcRes<NMAX>::max_smem, "CTAs per SM");
  static_assert(stg % 128 == 0 && tb % 16 == 0 && hr % 16 == 0 && b2hi % 16 == 0, "alignment");
};

// Shared memory of the prep kernel (one CTA per key head).  Up to 24 nodes
// (four CTAs per SM, bound by registers): staged q and k inputs, fp32 rows,
// Gram entries, tables; after the Gram the staging bytes hold the per-head
// T scratch and gate vectors of up to kPrepHeads value heads at a time.  At
// the large capacities (kCompact: two CTAs per SM, bound by shared memory)
// the regions are reused by phase:
//   * conv: staged q inputs in sq, the staged k inputs in the bytes of the q
//     rows of kqf (the k conv runs first, the q conv then overwrites them);
//     the accepted node's new conv window is kept aside in nw;
//   * after the conv: the Gram entries in sq, the fp32 rows still in kqf;
//   * after the Gram: the per-head scratch in kqf.
template <int NMAX>
struct PrepLayout {
  static constexpr int kPrepHeads = TcRes<NMAX>::prep_heads;
  using Ly = TcLayout<NMAX>;
  using CS = ConvStage<NMAX>;
  static constexpr int NP = round_up(NMAX, 4);
  static constexpr int KQP = kTcD + 4;                 // padded row pitch (bank spread)
  static constexpr int kRows = Ly::NC * KQP * 4;       // fp32 [NC][KQP]: k rows, then q rows
  static constexpr bool kCompact = TcRes<NMAX>::prep_ctas == 2;
  static_assert(!kCompact || CS::bytes <= NMAX * KQP * 4, "staged k inputs fit the q rows");
  static constexpr int sq = 0;                         // staged q inputs
  static constexpr int kqf = kCompact ? sq + CS::bytes : sq + 2 * CS::bytes;
  static constexpr int sk = kCompact ? kqf + NMAX * KQP * 4 : sq + CS::bytes;  // staged k inputs
  static constexpr int gr = kCompact ? sq : kqf + kRows;  // Gram entries
  static_assert(!kCompact || GramLayout<NMAX>::bytes <= CS::bytes, "Gram entries fit the staging");
  // per head chunk, after the Gram
  static constexpr int tf = kCompact ? kqf : 0;       // float [kPrepHeads][NMAX][TP]
  static constexpr int han = tf + kPrepHeads * NMAX * Ly::TP * 4;  // float [kPrepHeads][NP]
  static constexpr int hbn = han + kPrepHeads * NP * 4;
  static constexpr int hgam = hbn + kPrepHeads * NP * 4;
  static_assert(hgam + kPrepHeads * NP * 4 <= (kCompact ? kqf + kRows : 2 * CS::bytes),
                "head scratch fits");
  static constexpr int tb = kCompact ? kqf + kRows : gr + GramLayout<NMAX>::bytes;
  static constexpr int nw = tb + TabLayout<NMAX>::bytes;  // float [2][K-1][128]: q, k
  static constexpr int porig = nw + (kCompact ? 2 * (LBX_MAX_CONV_WIDTH - 1) * kTcD * 4 : 0);
  static constexpr int misc = porig + 4 * NP;
  static constexpr int bar = (misc + 64 + 7) & ~7;
  static constexpr int total = bar + 8;
  static_assert(sq % 128 == 0 && sk % 128 == 0, "TMA destinations");
  static_assert(total + 1024 <= 233472 / TcRes<NMAX>::prep_ctas, "prep CTAs per SM");
};

// Workspace layout of the tensor-core step: the tree tables of every
// request; one [K|Q] image per (layer, request, key head); one value-head
// record per tile (layer, request, value head), in tile order.
template <int NMAX>
__host__ __device__ inline size_t tc_tab_bytes(int Bq) {
  return ((size_t)Bq * TabLayout<NMAX>::bytes + 255) & ~(size_t)255;
}
template <int NMAX>
__host__ __device__ inline size_t tc_head_offset(int L, int Bq, int Hk) {
  return tc_tab_bytes<NMAX>(Bq) + (size_t)L * Bq * Hk * TcLayout<NMAX>::kB;
}
template <int NMAX>
__host__ __device__ inline size_t tc_workspace_bytes(int L, int Bq, int Hk, int Hv) {
  return tc_head_offset<NMAX>(L, Bq, Hk) + (size_t)L * Bq * Hv * HeadLayout<NMAX>::bytes;
}

struct TcArgs {
  StepArgs s;
  int n_tiles;        // L * Bq * Hv
  unsigned char *ws;  // workspace: tree tables, then per-key-head records
};

struct TcMaps {
  CUtensorMap state;  // [rows][128] fp32, box {32, 128}, 128-byte swizzle
  CUtensorMap x;      // [L*Bq*N][C] bf16, box {128, N}
  CUtensorMap cache;  // [L*n_slots*(K-1)][C] fp32, box {128, K-1} (K > 1)
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
// Byte offset of bf16 element (row, k) of a K-major operand with kp elements
// per row, no swizzle: core matrices of 8 rows x 16 bytes, 128 bytes apart
// along K, 8-row groups kp * 16 bytes apart.
__device__ __forceinline__ uint32_t plain_bf16(int kp, int row, int k) {
  return (uint32_t)((row >> 3) * kp * 16 + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// bf16 hi / lo split of x: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float x, uint16_t &hi, uint16_t &lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}
// The same for a pair, packed (a in the low half).
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}
// Conv-window sources of the persist: new row rr takes the (K-2-rr)-th
// ancestor of acc, or old cache row depth(acc)+1+rr where the path is short.
__device__ __forceinline__ void window_sources(int *dst, int K, int acc, const int *par) {
  int da = 0;
  for (int m = acc; m > 0; m = par[m]) ++da;
  for (int rr = 0; rr < K - 1; ++rr) {
    const int dist = K - 2 - rr;
    int w;
    if (dist <= da) {
      int m = acc;
      for (int q = 0; q < dist; ++q) m = par[m];
      w = m;
    } else {
      w = -1 - (da + 1 + rr);
    }
    dst[rr] = w;
  }
}

// Weights of 8 consecutive channels c0..c0+7 of a staged block, by window
// element: wsl[e][j] multiplies the j-th element of the window (tap K-1-j),
// 0 for j >= K.
template <int NMAX>
__device__ __forceinline__ void conv_weights8(float (&wsl)[8][LBX_MAX_CONV_WIDTH], int K,
                                              const unsigned char *cs, int c0) {
  using CS = ConvStage<NMAX>;
  const uint16_t *ws = reinterpret_cast<const uint16_t *>(cs + CS::w);
  if (K == LBX_MAX_CONV_WIDTH) {
    // the 8 channels' taps are 64 contiguous bytes: four 16-byte loads
    // (scalar loads at this lane stride conflict 8-way)
    const uint4 *w4 = reinterpret_cast<const uint4 *>(ws + c0 * LBX_MAX_CONV_WIDTH);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float t[8];
      unpack8(w4[q], t);  // channels c0 + 2q, c0 + 2q + 1, taps 0..3 each
#pragma unroll
      for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j) {
        wsl[2 * q][j] = t[LBX_MAX_CONV_WIDTH - 1 - j];
        wsl[2 * q + 1][j] = t[2 * LBX_MAX_CONV_WIDTH - 1 - j];
      }
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e)
#pragma unroll
    for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j)
      wsl[e][j] = j < K ? bf2f(ws[(c0 + e) * K + (K - 1 - j >= 0 ? K - 1 - j : 0)]) : 0.f;
}

// Conv + SiLU of 8 consecutive channels c0..c0+7 (within the staged block)
// of one node whose window rows are win[0..4) (>= 0: staged x row; < 0:
// staged cache row -1-w).  Loads use clamped, always-valid indices and the
// choice between the node row and the cache row is a select, so the unrolled
// body has no branches.
template <int NMAX>
__device__ __forceinline__ void conv8_staged(float (&out)[8], const int4 w4,
                                             const float (&wsl)[8][LBX_MAX_CONV_WIDTH],
                                             const unsigned char *cs, int c0) {
  using CS = ConvStage<NMAX>;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const int wj[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
  for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j) {
    const int row = wj[j];
    const int xr = row >= 0 ? row : 0;
    const int cr = row >= 0 ? 0 : -1 - row;
    float xn[8];
    unpack8(*reinterpret_cast<const uint4 *>(cs + CS::x + xr * kTcD * 2 + c0 * 2), xn);
    const float4 *cp = reinterpret_cast<const float4 *>(cs + CS::c + cr * kTcD * 4 + c0 * 4);
    const float4 lo = cp[0], hi = cp[1];
    const float xc[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(wsl[e][j], row >= 0 ? xn[e] : xc[e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) out[e] = silu_fast(acc[e]);
}

// conv8_staged for a node whose window lies inside the tree (every row
// >= 0): no cached-row loads, no selects.
template <int NMAX>
__device__ __forceinline__ void conv8_staged_tree(float (&out)[8], const int4 w4,
                                                  const float (&wsl)[8][LBX_MAX_CONV_WIDTH],
                                                  const unsigned char *cs, int c0) {
  using CS = ConvStage<NMAX>;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const int wj[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
  for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j) {
    float xn[8];
    unpack8(*reinterpret_cast<const uint4 *>(cs + CS::x + wj[j] * kTcD * 2 + c0 * 2), xn);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(wsl[e][j], xn[e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) out[e] = silu_fast(acc[e]);
}

// New conv-window entries of channel gc, from global memory: row rr takes
// src[rr] (>= 0: x row of the request; < 0: old cache row -1-src).  Every old
// value is read before any is written (the window is updated in place).
__device__ __forceinline__ void persist_channel_global(int gc, int K, int C, const int *src,
                                                       const uint16_t *x_lb, const float *cache_in,
                                                       float *cache_out) {
  float val[LBX_MAX_CONV_WIDTH - 1];
#pragma unroll
  for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr)
    if (rr < K - 1) {
      const int w = src[rr];
      val[rr] = w >= 0 ? bf2f(x_lb[(size_t)w * C + gc]) : cache_in[(size_t)(-1 - w) * C + gc];
    }
#pragma unroll
  for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr)
    if (rr < K - 1) cache_out[(size_t)rr * C + gc] = val[rr];
}

// Calls f(integral_constant<part>) for the run-time part index p < PARTS.
template <int PARTS, class F>
__device__ __forceinline__ void by_part(int p, F &&f) {
  if (p == 0) f(std::integral_constant<int, 0>{});
  else if (p == 1) f(std::integral_constant<int, 1>{});
  else if constexpr (PARTS > 2) {
    if (p == 2) f(std::integral_constant<int, 2>{});
    else f(std::integral_constant<int, 3>{});
  }
}

// Node values of part HF of a row (NMAX / parts nodes), as packed bf16
// pairs, hi and lo, into the A columns of MMA2 / MMA3 (hi at a2, lo at
// a2 + KP/2): part p writes the pairs of its nodes, the last part also the
// zero padding up to KP.
template <int NMAX, int HF>
__device__ __forceinline__ void store_pairs(uint32_t a2, const float *v) {
  using Ly = TcLayout<NMAX>;
  constexpr int PARTS = TcRes<NMAX>::parts;
  constexpr int NQ = NMAX / PARTS, KP = Ly::KP, KH = KP / 2;
  // the last part also zero-fills the padding columns up to KP
  constexpr int CNT = HF < PARTS - 1 ? NQ / 2 : (NQ + KP - NMAX) / 2, OFF = HF * NQ / 2;
  uint32_t ph[CNT], pl[CNT];
#pragma unroll
  for (int e = 0; e < CNT; ++e)
    split_bf16x2(2 * e < NQ ? v[2 * e] : 0.f, 2 * e + 1 < NQ ? v[2 * e + 1] : 0.f, ph[e], pl[e]);
  ptx::tmem_st_run<OFF, CNT>(a2, ph);
  ptx::tmem_st_run<OFF, CNT>(a2 + KH, pl);
}

// MMA1: S0 [K|Q]^T with B = [K|Q] (hi rows 0..NC-1, lo rows NC..2NC-1,
// K = 128, 128-byte swizzle) and S0 in TMEM (hi columns a, lo columns
// a + 64): pass 1, S0_hi x [B_hi | B_lo] (N = 2 NC), initialises 2 NC
// accumulator columns and pass 2, S0_lo x B_hi, adds into the first NC;
// column n of the product is the sum of columns n and NC + n.
template <int NMAX>
__device__ __forceinline__ void mma_kq(uint32_t d_tmem, uint32_t a, uint32_t b1) {
  using Ly = TcLayout<NMAX>;
  constexpr int NC = Ly::NC, R1 = Ly::R1;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const uint32_t idesc = pass == 0 ? ptx::idesc_bf16(128, 2 * NC) : ptx::idesc_bf16(128, NC);
#pragma unroll
    for (int ks = 0; ks < kTcD / 16; ++ks) {
      const uint32_t koff = (uint32_t)((ks >> 2) * (R1 * 128) + (ks & 3) * 32);
      ptx::mma_bf16_ts(d_tmem, a + (pass == 1 ? 64u : 0u) + 8u * ks, ptx::sdesc_sw128(b1 + koff),
                       idesc, (pass | ks) != 0);
    }
  }
}

template <int NMAX>
__global__ void __launch_bounds__(TcRes<NMAX>::threads, TcRes<NMAX>::ctas)
    gdn_step_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs T) {
  constexpr int NT = TcRes<NMAX>::threads, PARTS = TcRes<NMAX>::parts;
  using Ly = TcLayout<NMAX>;
  using CS = ConvStage<NMAX>;
  constexpr int NC = Ly::NC, R1 = Ly::R1, KP = Ly::KP, KH = KP / 2;
  const StepArgs &A = T.s;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *st = smem + Ly::stage;
  unsigned char *sg = smem + Ly::stg;
  unsigned char *B1 = smem + Ly::b1;  // [K|Q] hi rows 0..NC-1, lo rows NC..2NC-1
  unsigned char *B2hi = smem + Ly::b2hi;
  unsigned char *B2lo = smem + Ly::b2lo;
  using TL = TabLayout<NMAX>;
  using HL = HeadLayout<NMAX>;
  unsigned char *tb = smem + Ly::tb;
  const uint16_t *lofs = reinterpret_cast<const uint16_t *>(tb + TL::lofs);
  const int *win = reinterpret_cast<const int *>(tb + TL::win);
  const int *n2o = reinterpret_cast<const int *>(tb + TL::n2o);
  const int *crow = reinterpret_cast<const int *>(tb + TL::crow);
  const int *meta = reinterpret_cast<const int *>(tb + TL::meta);  // P, lanes, pairs
  unsigned char *hr = smem + Ly::hr;  // value-head record of the current tile
  const float *tw = reinterpret_cast<const float *>(hr + HL::tw);
  const float *an = reinterpret_cast<const float *>(hr + HL::an);
  const float *bn = reinterpret_cast<const float *>(hr + HL::bn);
  const float *gam = reinterpret_cast<const float *>(hr + HL::gam);
  const float *cpa = reinterpret_cast<const float *>(hr + HL::cpa);
  int *misc = reinterpret_cast<int *>(smem + Ly::misc);
  // misc[0] error flag, [3] TMEM base
  uint64_t *stage_bar = reinterpret_cast<uint64_t *>(smem + Ly::bars);
  uint64_t *stg_bar = stage_bar + 1;
  uint64_t *mma_bar = stage_bar + 2;
  uint64_t *rec_bar = stage_bar + 3;  // per-key-head record
  uint64_t *tab_bar = stage_bar + 4;  // per-request tables
  uint64_t *hr_bar = stage_bar + 5;   // per-tile value-head record

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const bool lead = tid == 0;  // issues the copies and the MMAs
  const int N = A.N, K = A.K, Hk = A.Hk, Hv = A.Hv, Bq = A.Bq;
  const int G = Hv / Hk;
  const int C = (2 * Hk + Hv) * kTcD;
  const uint32_t stg_bytes =
      (uint32_t)N * kTcD * 2 + (uint32_t)(K - 1) * kTcD * 4 + (uint32_t)kTcD * K * 2;

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
    ptx::mbar_init(stage_bar, 1);
    ptx::mbar_init(stg_bar, 1);
    ptx::mbar_init(mma_bar, 1);
    ptx::mbar_init(rec_bar, 1);
    ptx::mbar_init(tab_bar, 1);
    ptx::mbar_init(hr_bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t *>(&misc[3]), TcRes<NMAX>::tmem_cols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[3]);

  // tile -> (head in group, key-head group, key head, layer*Bq + request,
  // request, layer, value head)
  struct Tile {
    int hg, rest, kh, lbi, bq, l, h;
  };
  auto tile_of = [&](int t) {
    Tile x;
    x.hg = t % G;
    x.rest = t / G;
    x.kh = x.rest % Hk;
    x.lbi = x.rest / Hk;
    x.bq = x.lbi % Bq;
    x.l = x.lbi / Bq;
    x.h = x.kh * G + x.hg;
    return x;
  };
  // the tile after x (tiles are visited in order)
  auto next_tile = [&](Tile x) {
    if (++x.hg == G) {
      x.hg = 0;
      ++x.rest;
      if (++x.kh == Hk) {
        x.kh = 0;
        ++x.lbi;
        if (++x.bq == Bq) {
          x.bq = 0;
          ++x.l;
        }
      }
    }
    x.h = x.kh * G + x.hg;
    return x;
  };
  // cache slot of a request, read from global memory once per request
  struct SlotCache {
    int bq = -1, slot = 0;
  };
  auto slot_of = [&](SlotCache &c, int b) {
    if (b != c.bq) {
      c.bq = b;
      c.slot = A.slot[b];
    }
    return c.slot;
  };
  SlotCache lead_slots, tile_slots;
  // lead thread: copies into the stage and the staging buffer
  int n_state_loads = 0, n_stg_loads = 0;
  auto load_state = [&](const Tile &x) {
    const int srow = ((x.l * A.n_slots + slot_of(lead_slots, x.bq)) * Hv + x.h) * kTcD;
    ptx::mbar_arrive_expect_tx(stage_bar, kStageBytes);
    for (int a = 0; a < 4; ++a)
      ptx::tma_load_2d(st + a * (kStageBytes / 4), &maps.state, a * 32, srow, stage_bar);
    ++n_state_loads;
  };
  // conv inputs of the value head's channels
  auto load_block = [&](const Tile &x) {
    const int ch0 = (2 * Hk + x.h) * kTcD;
    const int crow0 = (x.l * A.n_slots + slot_of(lead_slots, x.bq)) * (K - 1);
    ptx::mbar_arrive_expect_tx(stg_bar, stg_bytes);
    ptx::tma_load_2d(sg + CS::x, &maps.x, ch0, x.lbi * N, stg_bar);
    if (K > 1) ptx::tma_load_2d(sg + CS::c, &maps.cache, ch0, crow0, stg_bar);
    ptx::bulk_load(sg + CS::w, A.conv_w + (size_t)x.l * C * K + (size_t)ch0 * K,
                   (uint32_t)kTcD * K * 2, stg_bar);
    ++n_stg_loads;
  };
  // the key head's [K|Q] image, the request's tree tables and the tile's
  // value-head record, from the workspace the prep kernel filled
  int n_rec_loads = 0, n_tab_loads = 0, n_hr_loads = 0, n_stores = 0;
  const unsigned char *imgs = T.ws + tc_tab_bytes<NMAX>(Bq);
  const unsigned char *heads = T.ws + tc_head_offset<NMAX>(A.L, Bq, Hk);
  auto load_rec = [&](const Tile &x) {
    ptx::mbar_arrive_expect_tx(rec_bar, (uint32_t)Ly::kB);
    ptx::bulk_load(B1, imgs + (size_t)x.rest * Ly::kB, (uint32_t)Ly::kB, rec_bar);
    ++n_rec_loads;
  };
  // the record of tile t: its used bytes when the tile's request is the one
  // whose tables are in shared memory (their lane count), else all of it
  auto load_hr = [&](int t, bool tables_match) {
    const uint32_t n = tables_match ? (uint32_t)HL::used(meta[1]) : (uint32_t)HL::bytes;
    ptx::mbar_arrive_expect_tx(hr_bar, n);
    ptx::bulk_load(hr, heads + (size_t)t * HL::bytes, n, hr_bar);
    ++n_hr_loads;
  };
  auto load_tab = [&](const Tile &x) {
    ptx::mbar_arrive_expect_tx(tab_bar, (uint32_t)TL::bytes);
    ptx::bulk_load(tb, T.ws + (size_t)x.bq * TL::bytes, (uint32_t)TL::bytes, tab_bar);
    ++n_tab_loads;
  };
  // phases waited for, the same count in every thread
  uint32_t stg_waits = 0, mma_waits = 0, rec_waits = 0, tab_waits = 0, hr_waits = 0;
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

  Tile cur = tile_of(t_begin);
  if (lead && count > 0) {
    // the state and the value-head inputs are not written by the prep
    // kernel: they load while it finishes; the workspace only after it
    load_state(cur);
    load_block(cur);
    ptx::wait_prerequisite_grid();
    load_tab(cur);
    load_rec(cur);
    load_hr(t_begin, false);
  }

  // state row r (= TMEM lane) and part pt of this thread; the row work of
  // nodes n0 .. n0 + NQ - 1 and of state columns pt * CPP .. + CPP - 1 is
  // this thread's
  const int quad = warp & 3, pt = warp >> 2;
  const int r = quad * 32 + (tid & 31);
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
  constexpr int NQ = NMAX / PARTS;                    // nodes per part
  constexpr int CPP = kTcD / PARTS;                   // state columns per part
  static_assert(NQ % 2 == 0 && CPP % 32 == 0, "node pairs, 32-column TMEM runs");
  const int n0 = pt * NQ;
  constexpr int LB = NQ <= 4 ? 4 : 8;  // accumulator columns per TMEM load

  int cur_req = -1, cur_group = -1;
  for (int it = 0; it < count; ++it) {
    const int t = t_begin + it;
    const Tile x = cur;
    const Tile nx = next_tile(x);
    cur = nx;
    const int bq = x.bq, l = x.l, h = x.h;
    const size_t lb = (size_t)x.lbi;
    const int slot_b = slot_of(tile_slots, bq);
    float *cache_o = A.conv_cache_out + ((size_t)l * A.n_slots + slot_b) * (K - 1) * C;

    // ================= tree tables (new request), record (new key head) =================
    if (bq != cur_req) {
      cur_req = bq;
      // [T | W] entries outside the (node, ancestor-or-self) pairs stay zero
      for (int idx = tid; idx < 2 * Ly::kB2 / 16; idx += NT)
        *reinterpret_cast<uint4 *>(B2hi + 16 * idx) = make_uint4(0u, 0u, 0u, 0u);
      wait_on(tab_bar, tab_waits);
    }
    if (x.rest != cur_group) {
      cur_group = x.rest;
      wait_on(rec_bar, rec_waits);
    }

    if (lead && it > 0) {
      ptx::bulk_wait_read_all();  // the previous tile's stores have read the stage
      load_state(x);
    }
    if (TcRes<NMAX>::ctas == 2 && lead && it + 1 < count) {
      // the next tile's slab into L2 while this tile runs, so that its copy
      // into the stage at the next tile's top reads L2 (at one CTA per SM,
      // 32 nodes and more, this measured slower and is left out)
      const int srow = ((nx.l * A.n_slots + slot_of(lead_slots, nx.bq)) * Hv + nx.h) * kTcD;
      ptx::prefetch_l2(A.state_in + (size_t)srow * kTcD, kStageBytes, ptx::policy_evict_last());
    }

    // ================= v of this row for this part's nodes (staged inputs) =================
    // before the slab is needed: the v conv covers the slab copy's latency
    wait_on(stg_bar, stg_waits);
    float vv[NQ];
    {
      const uint16_t *xs = reinterpret_cast<const uint16_t *>(sg + CS::x);
      const float *cs = reinterpret_cast<const float *>(sg + CS::c);
      float wslot[LBX_MAX_CONV_WIDTH];  // weight of window element j
      {
        const uint16_t *ws = reinterpret_cast<const uint16_t *>(sg + CS::w) + r * K;
#pragma unroll
        for (int j = 0; j < LBX_MAX_CONV_WIDTH; ++j)
          wslot[j] = j < K ? bf2f(ws[K - 1 - j >= 0 ? K - 1 - j : 0]) : 0.f;
      }
      // v of this row for node n0 + i, window element j weighted by wslot[j]
      // (element 0 is the node's own input row, never a cached row)
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const int4 w4 = *reinterpret_cast<const int4 *>(win + 4 * (n0 + i));
        const int wj[4] = {w4.x, w4.y, w4.z, w4.w};
        float y = wslot[0] * bf2f(xs[wj[0] * kTcD + r]);
#pragma unroll
        for (int j = 1; j < LBX_MAX_CONV_WIDTH; ++j) {
          const int w = wj[j];
          const float xn = bf2f(xs[(w >= 0 ? w : 0) * kTcD + r]);
          const float xc = cs[(w >= 0 ? 0 : -1 - w) * kTcD + r];
          y = fmaf(wslot[j], w >= 0 ? xn : xc, y);
        }
        vv[i] = silu_fast(y);
      }
      // this row's value channel of the conv window (only this tile reads it)
      if (pt == 0) {
#pragma unroll
        for (int rr = 0; rr < LBX_MAX_CONV_WIDTH - 1; ++rr)
          if (rr < K - 1) {
            const int w = crow[rr];
            const float v = w >= 0 ? bf2f(xs[w * kTcD + r]) : cs[(-1 - w) * kTcD + r];
            cache_o[(size_t)rr * C + (2 * Hk + h) * kTcD + r] = v;
          }
      }
    }
    // ================= [T | W] of this value head =================
    wait_on(hr_bar, hr_waits);
    ptx::named_sync(1, NT);  // staging consumed; zero-filled [T|W] (new request) before the scatter
    if (lead && it + 1 < count) load_block(nx);
    const float gacc = reinterpret_cast<const float *>(hr + HL::gacc)[0];
    {
      const int nl = meta[1], nl4 = HL::lanes4(nl);
      for (int lane = tid; lane < nl; lane += NT) {
        const uint32_t o = lofs[lane];
        uint16_t th, tl, wh, wl;
        split_bf16(tw[lane], th, tl);
        split_bf16(tw[nl4 + lane], wh, wl);
        *reinterpret_cast<uint16_t *>(B2hi + o) = th;
        *reinterpret_cast<uint16_t *>(B2lo + o) = tl;
        *reinterpret_cast<uint16_t *>(B2hi + o + Ly::kWOff) = wh;
        *reinterpret_cast<uint16_t *>(B2lo + o + Ly::kWOff) = wl;
      }
    }
    ptx::fence_proxy_async();

    // ================= S0 -> tensor memory (bf16 hi / lo) =================
    if (!ptx::mbar_wait(stage_bar, (uint32_t)(it & 1))) {
      if (A.status) *A.status = LBX_ETIMEOUT;
      bad = true;
    }
    {
      // this thread's CPP columns of the row, 32 at a time: hi into A
      // columns pt * CPP / 2 .., lo 64 columns further
#pragma unroll
      for (int c = 0; c < CPP / 32; ++c) {
        uint32_t vh[16], vl[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x4 =
              *reinterpret_cast<const float4 *>(st + sw128_f32(kTcD, r, pt * CPP + 32 * c + 4 * q));
          split_bf16x2(x4.x, x4.y, vh[2 * q], vl[2 * q]);
          split_bf16x2(x4.z, x4.w, vh[2 * q + 1], vl[2 * q + 1]);
        }
        ptx::tmem_st16(tq + Ly::cA1 + pt * (CPP / 2) + 16 * c, vh);
        ptx::tmem_st16(tq + Ly::cA1 + 64 + pt * (CPP / 2) + 16 * c, vl);
      }
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    if (__syncthreads_or(bad)) {  // ---------------------------------------------- S1
      aborted = true;
      break;
    }

    if (lead) {
      // MMA1: [S0 k | S0 q] = S0 [K|Q]^T over K = 128
      ptx::tc_fence_after();
      mma_kq<NMAX>(tmem + Ly::cD1, tmem + Ly::cA1, ptx::smem_u32(B1));
      ptx::mma_commit(mma_bar);
    }


    // ================= rhs -> tensor memory =================
    // Accumulator columns are read in aligned blocks of LB covering this
    // part's nodes; node N0 + i sits at position SH + i of the block.
    wait_on(mma_bar, mma_waits);
    ptx::tc_fence_after();
    float oq[NQ];
    auto rhs_part = [&](auto pc) {
      constexpr int HF = decltype(pc)::value;
      constexpr int N0 = HF * NQ, B0 = N0 / LB * LB, SH = N0 - B0;
      constexpr int NL = round_up(SH + NQ, LB);
      // rhs_n = b_n v_n - b_n a_n gamma_p S0 k_n (0 for padding nodes)
      float rhs[NQ];
      // accumulator columns in pieces of CH * LB (all at once for small
      // parts; 8 columns at a time for the large ones, to bound registers)
      constexpr int CH = NQ > 12 ? 1 : NL / LB;
      static_assert(CH == NL / LB || SH == 0, "chunked parts start aligned");
#pragma unroll
      for (int c0 = 0; c0 < NL / LB; c0 += CH) {
        float k_hi[CH * LB], k_lo[CH * LB], q_hi[CH * LB], q_lo[CH * LB];
#pragma unroll
        for (int b = 0; b < CH; ++b) {
          const int cb = B0 + (c0 + b) * LB;
          ptx::tmem_ld_w<LB>(tq + Ly::cD1 + cb, k_hi + b * LB);
          ptx::tmem_ld_w<LB>(tq + Ly::cD1 + NC + cb, k_lo + b * LB);
          ptx::tmem_ld_w<LB>(tq + Ly::cD1 + NMAX + cb, q_hi + b * LB);
          ptx::tmem_ld_w<LB>(tq + Ly::cD1 + NC + NMAX + cb, q_lo + b * LB);
        }
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < CH * LB; ++e) {
          const int i = c0 * LB + e - SH;  // node N0 + i
          if (i >= 0 && i < NQ) {
            const int n = N0 + i;
            const float ag = an[n] * gam[n];
            rhs[i] = bn[n] * fmaf(-ag, k_hi[e] + k_lo[e], vv[i]);
            oq[i] = ag * (q_hi[e] + q_lo[e]);
          }
        }
      }
      store_pairs<NMAX, HF>(tq + Ly::cA2, rhs);
    };
    by_part<PARTS>(pt, rhs_part);
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    if (__syncthreads_or(bad)) {  // ---------------------------------------------- S2
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

    // ================= path deltas -> tensor memory =================
    wait_on(mma_bar, mma_waits);
    ptx::tc_fence_after();
    auto dl_part = [&](auto pc) {
      constexpr int HF = decltype(pc)::value;
      constexpr int N0 = HF * NQ, B0 = N0 / LB * LB, SH = N0 - B0;
      constexpr int NL = round_up(SH + NQ, LB);
      constexpr int CH = NQ > 12 ? 1 : NL / LB;
      float dl[NQ];
#pragma unroll
      for (int c0 = 0; c0 < NL / LB; c0 += CH) {
        float dd[CH * LB];
#pragma unroll
        for (int b = 0; b < CH; ++b)
          ptx::tmem_ld_w<LB>(tq + Ly::cD2 + B0 + (c0 + b) * LB, dd + b * LB);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < CH * LB; ++e) {
          const int i = c0 * LB + e - SH;  // node N0 + i
          if (i >= 0 && i < NQ) dl[i] = cpa[N0 + i] * dd[e];
        }
      }
      store_pairs<NMAX, HF>(tq + Ly::cA2, dl);
    };
    by_part<PARTS>(pt, dl_part);
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    if (__syncthreads_or(bad)) {  // ---------------------------------------------- S3
      aborted = true;
      break;
    }
    if (lead) {
      // MMA3: sum_j c_j delta_j k_j^T over the path rows of operand K,
      // read N-major, three passes over K = KP
      ptx::tc_fence_after();
      constexpr uint32_t idesc = ptx::idesc_bf16_bmn(128, kTcD);
      const uint32_t b1_a = ptx::smem_u32(B1);
      uint32_t accum = 0;
#pragma unroll 1
      for (int pass = 0; pass < 3; ++pass) {
        const uint32_t a_col = Ly::cA2 + (pass == 2 ? KH : 0);
        const uint32_t b_base = b1_a + (pass == 1 ? (uint32_t)NC * 128u : 0u);  // lo rows
#pragma unroll
        for (int ks = 0; ks < KP / 16; ++ks) {
          ptx::mma_bf16_ts(tmem + Ly::cA1, tmem + a_col + 8 * ks,
                           ptx::sdesc(b_base + 2048u * ks, (uint32_t)R1 * 128u, 1024u, 2u), idesc,
                           accum);
          accum = 1;
        }
      }
      ptx::mma_commit(mma_bar);
      // every thread has passed its last read of this tile's value-head
      // record (S3): bring in the next tile's
      if (it + 1 < count) load_hr(t + 1, nx.bq == bq);
    }

    // ================= o = diag(a gamma_p) S0 q + W rhs, while MMA3 runs =================
    // (MMA3 writes the S0 columns; W rhs sits in the MMA2 accumulator)
    ptx::tc_fence_after();
    auto o_part = [&](auto pc) {
      constexpr int HF = decltype(pc)::value;
      constexpr int N0 = HF * NQ, B0 = N0 / LB * LB, SH = N0 - B0;
      constexpr int NL = round_up(SH + NQ, LB);
      constexpr int CH = NQ > 12 ? 1 : NL / LB;
      float *o_base = A.o + (lb * N) * (size_t)Hv * kTcD + (size_t)h * kTcD + r;
#pragma unroll
      for (int c0 = 0; c0 < NL / LB; c0 += CH) {
        float wr[CH * LB];
#pragma unroll
        for (int b = 0; b < CH; ++b)
          ptx::tmem_ld_w<LB>(tq + Ly::cD2 + NMAX + B0 + (c0 + b) * LB, wr + b * LB);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < CH * LB; ++e) {
          const int i = c0 * LB + e - SH;  // node N0 + i
          if (i >= 0 && i < NQ && N0 + i < N)
            __stcs(o_base + (size_t)n2o[N0 + i] * Hv * kTcD, oq[i] + wr[e]);
        }
      }
    };
    by_part<PARTS>(pt, o_part);
    if (lead && it + 1 < count && nx.rest != x.rest) {
      // the next tile starts a key head: its record replaces this one once
      // MMA3 (the last reader of the operand) has completed
      if (ptx::mbar_wait(mma_bar, mma_waits & 1u)) load_rec(nx);
    }

    // ================= accepted state (gamma_acc S0 + MMA3) -> global memory =================
    // formed in place over this thread's bytes of the staged S0 (the box
    // layout the copies use), then stored by TMA; the next slab follows
    wait_on(mma_bar, mma_waits);
    ptx::tc_fence_after();
    {
      const int sw = r & 7;
#pragma unroll
      for (int c = 0; c < CPP / 32; ++c) {
        const int box = (CPP * pt) / 32 + c;
        unsigned char *row = st + box * (kStageBytes / 4) + r * 128;
        float d[32];
        ptx::tmem_ld32(tq + Ly::cA1 + 32 * box, d);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 *p4 = reinterpret_cast<float4 *>(row + ((q ^ sw) << 4));
          const float4 s4 = *p4;
          *p4 = make_float4(fmaf(gacc, s4.x, d[4 * q]), fmaf(gacc, s4.y, d[4 * q + 1]),
                            fmaf(gacc, s4.z, d[4 * q + 2]), fmaf(gacc, s4.w, d[4 * q + 3]));
        }
      }
    }
    ptx::fence_proxy_async();  // the staged rows, for the TMA stores
    ptx::tc_fence_before();
    if (__syncthreads_or(bad)) {  // ---------------------------------------------- S4
      aborted = true;
      break;
    }
    if (lead) {
      const int srow = ((l * A.n_slots + slot_b) * Hv + h) * kTcD;
      for (int a = 0; a < 4; ++a)
        ptx::tma_store_2d(&maps.state, a * 32, srow, st + a * (kStageBytes / 4));
      ptx::bulk_commit();
      ++n_stores;
      // the next slab is loaded once the stores have read the stage, at the
      // next tile's top (so that the issuing thread does not stall here
      // while the stores drain)
      if (it + 1 < count && nx.bq != bq) load_tab(nx);
    }
  }

  // ---- drain: copies still in flight after an abort ----
  if (lead && aborted) {
    if (n_state_loads > 0) (void)ptx::mbar_wait(stage_bar, (uint32_t)((n_state_loads - 1) & 1));
    if (n_stg_loads > 0) (void)ptx::mbar_wait(stg_bar, (uint32_t)((n_stg_loads - 1) & 1));
    if (n_rec_loads > 0) (void)ptx::mbar_wait(rec_bar, (uint32_t)((n_rec_loads - 1) & 1));
    if (n_tab_loads > 0) (void)ptx::mbar_wait(tab_bar, (uint32_t)((n_tab_loads - 1) & 1));
    if (n_hr_loads > 0) (void)ptx::mbar_wait(hr_bar, (uint32_t)((n_hr_loads - 1) & 1));
  }
  // the state stores complete before the CTA leaves
  if (lead && n_stores > 0) ptx::bulk_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TcRes<NMAX>::tmem_cols);
  }
}

}  // namespace lbx
