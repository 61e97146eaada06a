// tree_attn.cu -- tree-masked attention of the full-attention layers on the
// tensor cores (sm_103a): lbx_attn_workspace_size, lbx_tree_attention.
//
// In the verify forward every draft node's query attends to the request's
// cached context and to the tree nodes on its own root path (Lucebox hub
// README: DDTree verifies the whole tree in one target forward, "Algorithms
// used"; the full-attention layers keep a KV cache, "--max-ctx N", with full
// attention by default, "--fa-window N" = 0).  For request b, KV head g and
// the G = Hq/Hkv query heads that read it, the queries of all (head, node)
// pairs share every key, so they form the rows of one matrix:
//
//   S = Q K^T (rows = (head, node) pairs, columns = keys)  -- tensor cores
//   online softmax over the key blocks, row by row         -- one thread per row
//   O += P V                                               -- tensor cores
//
// The work is the list of (row tile, key block) pairs: per (layer, request,
// KV head, row tile) the request's context blocks of 64 keys, then one block
// with the tree's own keys under the ancestor mask.  Row tiles hold at most
// 128 rows (hp heads x N nodes; 6 x 22 = 132 at budget 22 gives two tiles of
// 66).  A persistent grid (one CTA per SM) is cut into groups of `tiles`
// consecutive CTAs; the groups split the list of (layer, request, KV head,
// key block) into equal contiguous ranges, counted from the actual context
// lengths, and the CTAs of a group take one row tile each of the same range,
// so each K/V block is read from DRAM once and from L2 by the group's other
// CTAs.  A range covers a few (layer, request, KV head) groups, and a row
// tile is covered by one, two or three CTAs.  Each CTA writes the
// unnormalised partial (running max m, sum l, O) of every row tile it covers
// to the workspace; the last of a row tile's CTAs to finish merges them.
//
// Per CTA: the Q tile (128 rows x 256 bf16) stays in tensor memory, written
// row by row by the softmax threads at the start of each segment; K and V
// blocks of 64 keys arrive by TMA (four K and three V blocks in flight); S and
// P of a block share one of two 64-column TMEM buffers (the softmax threads
// overwrite S with P after the max exchange), and O takes 256 columns.  The
// issuing thread computes S = Q K^T with A = Q from tensor memory and O += P V
// with A = P from tensor memory.  P is split into bf16 hi + lo and
// multiplies V twice, so the product keeps ~2^-17 of relative precision (Q,
// K and V are exact bf16 inputs, accumulation is fp32).  The softmax
// reference point moves only when a block's maximum exceeds it by more than
// 2^8, so O is rescaled (a pass over its 256 columns) rarely; the result is
// the same softmax, referenced to a different maximum.  Every mbarrier wait
// is bounded; a CTA whose wait gives up reports LBX_ETIMEOUT, still counts
// itself in (with an empty partial) and drains its copies before leaving.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <cstring>
#include <mutex>

#include "lbx.h"
#include "tc_ptx.cuh"

namespace lbx {
namespace attn {

constexpr int kDh = LBX_ATTN_HEAD_DIM;  // head dimension (256)
constexpr int kRows = 128;              // query rows per CTA = TMEM lanes
constexpr int kKB = 64;                 // keys per block
constexpr int kKStages = 4;             // K blocks in flight
constexpr int kVStages = 3;             // V blocks in flight
constexpr int kMaxNodes = LBX_ATTN_MAX_NODES;
// Largest persistent grid (one CTA per SM; a GPU with more SMs uses this
// many); the workspace holds one partial per (CTA, row tile) piece, at most
// kMaxCtas + row tiles of them.
constexpr int kMaxCtas = 160;

// shared memory: K stages, V stages, ancestor masks, ints, mbarriers (the Q
// tile lives in tensor memory)
constexpr int kKVAtom = kKB * 128;                 // one 64-column atom of a block
constexpr int kKBytes = (kDh / 64) * kKVAtom;      // 32 KB: one K (or V) block
constexpr int kSmemK = 0;
constexpr int kSmemV = kSmemK + kKStages * kKBytes;
constexpr int kSmemAnc = kSmemV + kVStages * kKBytes;      // uint64 [64]
constexpr int kSmemRed = kSmemAnc + kMaxNodes * 8;        // float [2][128]
constexpr int kSmemMisc = kSmemRed + 2 * kRows * 4;       // int [16]
constexpr int kNBars = kKStages + kVStages + 6;           // k, v, s[2], o[2], p[2]
constexpr int kSmemBars = kSmemMisc + 64;                 // uint64 [kNBars]
constexpr int kSmemTotal = kSmemBars + kNBars * 8;
// threads: 8 softmax warps (two threads per row) and one issuing warp
constexpr int kSoftmaxThreads = 2 * kRows;
constexpr int kThreads = kSoftmaxThreads + 32;
static_assert(kSmemTotal <= 227 * 1024, "shared memory");
static_assert(kSmemK % 1024 == 0 && kSmemV % 1024 == 0 && kKBytes % 1024 == 0,
              "swizzled operands");
// tensor memory columns: the Q tile (operand A of S = Q K^T: row = lane,
// bf16 pairs along dh); S and P of block q in buffer q & 1 (the softmax
// threads read S, meet at the max exchange, then overwrite it with P: bf16 hi
// in the first 32 columns, lo in the other 32, operand A of O += P V); O
constexpr uint32_t kColQ = 0;     // 128 columns
constexpr uint32_t kColSP = 128;  // two 64-column buffers
constexpr uint32_t kColO = 256;   // 256 columns
constexpr uint32_t kTmemCols = 512;
static_assert(kColQ + kDh / 2 <= kColSP && kColSP + 2 * kKB <= kColO &&
                  kColO + kDh <= kTmemCols,
              "tensor memory");

// Row tiles (host and device compute the same).
struct Geo {
  int G;         // query heads per KV head
  int tiles;     // row tiles per (layer, request, KV head)
  int hp;        // heads per row tile (the last may hold fewer)
  long long gt;  // (layer, request, KV head, tile) groups
  int rows_cap;  // hp * N
};

__host__ __device__ inline Geo geometry(int L, int Bq, int N, int Hq, int Hkv) {
  Geo g;
  g.G = Hq / Hkv;
  g.tiles = 1;
  while (((g.G + g.tiles - 1) / g.tiles) * N > kRows) ++g.tiles;
  g.hp = (g.G + g.tiles - 1) / g.tiles;
  g.tiles = (g.G + g.hp - 1) / g.hp;
  g.gt = (long long)L * Bq * Hkv * g.tiles;
  g.rows_cap = g.hp * N;
  return g;
}

// Floats of one partial: m[128], l[128], then O rows of 256.
__host__ __device__ inline size_t unit_floats(const Geo &g) {
  return 2 * (size_t)kRows + (size_t)g.rows_cap * kDh;
}
__host__ __device__ inline size_t part_bytes(const Geo &g) {
  return (((size_t)g.gt + kMaxCtas + g.tiles) * unit_floats(g) * 4 + 255) & ~(size_t)255;
}

struct Args {
  int L, Bq, N, Hq, Hkv, T;
  Geo geo;
  float scale_log2;  // scale * log2(e): the softmax runs in base 2
  const uint16_t *q;
  const int32_t *ctx_len, *parent;
  float *o;
  float *part;
  unsigned int *counters;  // one per (layer, request, KV head, tile)
  int32_t *status;
};

struct Maps {
  CUtensorMap kc, vc;  // caches as (dh, Hkv, L*Bq*T), box (64, 1, 64), 128-byte swizzle
  CUtensorMap kt, vt;  // tree keys / values as (dh, Hkv, L*Bq*N)
};

__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// One plain arrival on an mbarrier (release semantics for this thread's
// earlier memory operations).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}

// 2^x on the hardware exponential unit (x <= 0 here; -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two threads per row: thread (row r, half hf) handles keys 32 hf .. 32 hf +
// 31 of every block and columns 128 hf .. 128 hf + 127 of O.  Warps w and w+4
// share TMEM lane quadrant w & 3.
constexpr int kHalfKeys = kKB / 2;
constexpr int kHalfCols = kDh / 2;

// Blocks of request b's row tiles: its context blocks and the tree block.
__device__ __forceinline__ int blocks_of(const int32_t *ctx_len, int b) {
  return (ctx_len[b] + kKB - 1) / kKB + 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    tree_attn_kernel(const __grid_constant__ Maps maps, const Args A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Geo &g = A.geo;
  const int N = A.N, Bq = A.Bq, Hkv = A.Hkv, tiles = g.tiles;
  int *misc = reinterpret_cast<int *>(smem + kSmemMisc);  // [0] TMEM base, [1] last CTA
  uint64_t *anc = reinterpret_cast<uint64_t *>(smem + kSmemAnc);
  float *red = reinterpret_cast<float *>(smem + kSmemRed);  // [2][kRows] per-half values
  uint64_t *k_bar = reinterpret_cast<uint64_t *>(smem + kSmemBars);  // [kKStages]
  uint64_t *v_bar = k_bar + kKStages;                                 // [kVStages]
  uint64_t *s_bar = v_bar + kVStages;                                 // [2]
  uint64_t *o_bar = s_bar + 2;                                        // [2]
  uint64_t *p_full = o_bar + 2;  // [2] the softmax threads have stored P (256 arrivals)

  // ---- whole-batch validation (the same verdict in every CTA) ----
  {
    int bad_in = 0;
    for (int i = tid; i < Bq * N; i += kThreads) {
      const int n = i % N, p = A.parent[i];
      if (n == 0 ? p != -1 : (p < 0 || p >= n)) bad_in = 1;
    }
    for (int i = tid; i < Bq; i += kThreads)
      if (A.ctx_len[i] < 0 || A.ctx_len[i] > A.T) bad_in = 1;
    if (__syncthreads_or(bad_in)) {
      if (tid == 0 && A.status) *A.status = LBX_ETREE;
      return;
    }
  }

  // ---- the flattened work list and this CTA group's range of it ----
  long long s_all = 0;  // blocks of one (layer, KV head) across the requests
  for (int b = 0; b < Bq; ++b) s_all += blocks_of(A.ctx_len, b);
  const long long per_l = (long long)Hkv * s_all;
  const long long total = (long long)A.L * per_l;
  // groups of `tiles` CTAs, at most one group per block, so that every
  // group's range is non-empty
  long long P = (long long)gridDim.x / tiles;
  if (P > total) P = total;
  const long long cg = blockIdx.x / tiles;
  const int tile = (int)(blockIdx.x - cg * tiles);
  if (cg >= P) return;
  const long long x_begin = total * cg / P, x_end = total * (cg + 1) / P;
  auto owner = [&](long long x) { return ((x + 1) * P - 1) / total; };

  // ---- set-up ----
  if (tid == 0) {
    for (int i = 0; i < kNBars - 2; ++i) ptx::mbar_init(k_bar + i, 1);
    for (int i = kNBars - 2; i < kNBars; ++i) ptx::mbar_init(k_bar + i, kSoftmaxThreads);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t *>(&misc[0]), kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int quad = warp & 3, hf = (warp >> 2) & 1;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);  // this warp's lane quadrant
  const int r = quad * 32 + lane;
  // warps 0-7 run the softmax (two threads per row); lane 0 of warp 8 issues
  // every copy and MMA and meets them through mbarriers only
  const bool softmax = tid < kSoftmaxThreads;
  const bool issuer = tid == kSoftmaxThreads;

  // descriptors of stage 0; the others are fixed offsets (added to the
  // 16-byte address field)
  const uint64_t kdesc0 = ptx::sdesc_sw128(ptx::smem_u32(smem + kSmemK));
  const uint64_t vdesc0 =
      ptx::sdesc(ptx::smem_u32(smem + kSmemV), (uint32_t)kKVAtom, 1024u, 2u);

  // Blocks are numbered q = 0, 1, ... across this CTA's segments; stages,
  // buffers and mbarrier phases follow q.
  long long q0 = 0;
  int n_kloads = 0, n_vloads = 0, n_mma1 = 0, n_mma2 = 0;  // issued by the issuer
  bool bad = false, aborted = false;

  // after an abort a CTA still walks its range, writing empty partials and
  // counting itself in, so that every group's counter completes and re-arms
  long long x = x_begin;
  while (x < x_end) {
    // ---- locate block x: layer, request, KV head, tile, block of the group ----
    const int l = (int)(x / per_l);
    long long rem = x - (long long)l * per_l, base_b = 0;
    int b = 0, nbr = blocks_of(A.ctx_len, 0);
    while (rem >= (long long)Hkv * nbr) {
      rem -= (long long)Hkv * nbr;
      base_b += (long long)Hkv * nbr;
      ++b;
      nbr = blocks_of(A.ctx_len, b);
    }
    const int kvh = (int)(rem / nbr), blk0 = (int)(rem - (long long)kvh * nbr);
    const int lb = l * Bq + b;
    const long long kvg = (long long)lb * Hkv + kvh;  // (layer, request, KV head)
    const long long gidx = kvg * tiles + tile;        // its row tile of this CTA
    const long long g_first = (long long)l * per_l + base_b + (long long)kvh * nbr;
    const int blk1 = (int)((x_end - g_first < nbr ? x_end - g_first : nbr));  // end of segment
    x = g_first + blk1;
    const int ctx = A.ctx_len[b];
    const int nctx = nbr - 1;                 // context blocks of the request
    const int nb = aborted ? 0 : blk1 - blk0;  // blocks of this segment
    const bool has_tree = blk1 == nbr;        // the segment ends with the tree block
    const int h0 = tile * g.hp;
    const int hp_t = g.G - h0 < g.hp ? g.G - h0 : g.hp;
    const int rows = hp_t * N;
    const bool real_row = softmax && r < rows;
    const int n_row = real_row ? r - (r / N) * N : 0;

    // ---- Q tile, ancestor masks (all of this segment's earlier MMAs are done) ----
    if (has_tree && tid < N) {  // ancestor-or-self mask of node tid
      uint64_t m = 0;
      int j = tid;
      for (int s = 0; s < kMaxNodes && j >= 0; ++s) {
        m |= 1ull << j;
        j = A.parent[(size_t)b * N + j];
      }
      anc[tid] = m;
    }
    if (softmax) {
      // this thread's half of its row's q (zero on padding rows) -> the Q
      // tile in tensor memory, bf16 pairs along dh
      const uint4 *qg = reinterpret_cast<const uint4 *>(A.q);
      const bool rv = r < rows;
      size_t qrow = 0;
      if (rv) {
        const int hl = r / N, n = r - hl * N;
        const int hq = kvh * g.G + h0 + hl;
        qrow = (((size_t)lb * N + n) * A.Hq + hq) * (kDh / 8) + hf * (kDh / 16);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = rv ? qg[qrow + c * 8 + e] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * e] = v.x;
          w[4 * e + 1] = v.y;
          w[4 * e + 2] = v.z;
          w[4 * e + 3] = v.w;
        }
        ptx::tmem_st32(tq + kColQ + (uint32_t)(hf * (kDh / 4) + 32 * c), w);
      }
      ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint64_t my_anc = has_tree && real_row ? anc[n_row] : 0ull;

    // block i of the segment: context block blk0 + i, or the tree block
    auto z_of = [&](int i) {
      const int jb = blk0 + i;
      return jb < nctx ? lb * A.T + jb * kKB : lb * N;
    };
    auto map_k = [&](int i) { return blk0 + i < nctx ? &maps.kc : &maps.kt; };
    auto map_v = [&](int i) { return blk0 + i < nctx ? &maps.vc : &maps.vt; };
    auto load_k = [&](int i) {
      const long long q = q0 + i;
      const int s = (int)(q % kKStages);
      unsigned char *kd = smem + kSmemK + s * kKBytes;
      ptx::mbar_arrive_expect_tx(&k_bar[s], (uint32_t)kKBytes);
#pragma unroll
      for (int a = 0; a < kDh / 64; ++a)
        ptx::tma_load_3d(kd + a * kKVAtom, map_k(i), a * 64, kvh, z_of(i), &k_bar[s]);
      ++n_kloads;
    };
    auto load_v = [&](int i) {
      const long long q = q0 + i;
      const int s = (int)(q % kVStages);
      unsigned char *vd = smem + kSmemV + s * kKBytes;
      ptx::mbar_arrive_expect_tx(&v_bar[s], (uint32_t)kKBytes);
#pragma unroll
      for (int a = 0; a < kDh / 64; ++a)
        ptx::tma_load_3d(vd + a * kKVAtom, map_v(i), a * 64, kvh, z_of(i), &v_bar[s]);
      ++n_vloads;
    };
    // S[q & 1] = Q K^T of segment block i: M = 128, N = 64 keys, K = 256
    auto mma1 = [&](int i) {
      const long long q = q0 + i;
      const uint64_t kd = kdesc0 + (uint64_t)(((q % kKStages) * kKBytes) >> 4);
      constexpr uint32_t idesc = ptx::idesc_bf16(128, kKB);
      const uint32_t d = tmem + kColSP + (uint32_t)(q & 1) * kKB;
#pragma unroll
      for (int ks = 0; ks < kDh / 16; ++ks) {
        const uint64_t bo = (uint64_t)(((ks >> 2) * kKVAtom + (ks & 3) * 32) >> 4);
        ptx::mma_bf16_ts(d, tmem + kColQ + 8u * ks, kd + bo, idesc, ks > 0 ? 1u : 0u);
      }
      ptx::mma_commit(&s_bar[q & 1]);
      ++n_mma1;
    };
    // O += P V of segment block i: A = P (TMEM, hi then lo), B = the V block
    // read MN-major (dh contiguous in 64-column atoms, 8-key groups 1024 apart)
    auto mma2 = [&](int i, bool acc) {
      const long long q = q0 + i;
      const uint64_t vd = vdesc0 + (uint64_t)(((q % kVStages) * kKBytes) >> 4);
      constexpr uint32_t idesc = ptx::idesc_bf16_bmn(128, kDh);
      const uint32_t pc = tmem + kColSP + (uint32_t)(q & 1) * kKB;
      uint32_t accum = acc ? 1u : 0u;
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int ks = 0; ks < kKB / 16; ++ks) {
          ptx::mma_bf16_ts(tmem + kColO, pc + pass * (kKB / 2) + ks * 8,
                           vd + (uint64_t)(ks * 2048 >> 4), idesc, accum);
          accum = 1u;
        }
      ptx::mma_commit(&o_bar[q & 1]);
      ++n_mma2;
    };

    float m_run = -INFINITY, l_run = 0.f;  // base-2 running max; this half's sum
    if (issuer) {
      // ---- the issuing thread: copies and MMAs in block order ----
      if (nb > 0) {
        for (int i = 0; i < nb && i < kKStages; ++i) load_k(i);
        for (int i = 0; i < nb && i < kVStages; ++i) load_v(i);
        if (!ptx::mbar_wait(&k_bar[q0 % kKStages], (uint32_t)((q0 / kKStages) & 1))) bad = true;
        if (!bad) mma1(0);
      }
      for (int i = 0; i < nb && !bad; ++i) {
        const long long q = q0 + i;
        // the next block's scores, into the other buffer once the product
        // that read its P (block i - 1; earlier segments are done) is done
        if (i + 1 < nb) {
          if (!ptx::mbar_wait(&k_bar[(q + 1) % kKStages], (uint32_t)(((q + 1) / kKStages) & 1)))
            bad = true;
          if (i >= 1 && !bad &&
              !ptx::mbar_wait(&o_bar[(q - 1) & 1], (uint32_t)(((q - 1) >> 1) & 1)))
            bad = true;
          if (!bad) mma1(i + 1);
        }
        // K of this block is free once its S is complete: block i + 3 there
        if (i + kKStages < nb) {
          if (!bad && !ptx::mbar_wait(&s_bar[q & 1], (uint32_t)((q >> 1) & 1))) bad = true;
          if (!bad) load_k(i + kKStages);
        }
        // this block's P, then O += P V
        if (!bad && !ptx::mbar_wait(&p_full[q & 1], (uint32_t)((q >> 1) & 1))) bad = true;
        if (!bad && !ptx::mbar_wait(&v_bar[q % kVStages], (uint32_t)((q / kVStages) & 1)))
          bad = true;
        if (bad) break;
        ptx::tc_fence_after();
        mma2(i, i > 0);
        // the previous product is done: its V stage takes block i - 1 + kVStages
        if (i >= 1 && i - 1 + kVStages < nb) {
          if (!ptx::mbar_wait(&o_bar[(q - 1) & 1], (uint32_t)(((q - 1) >> 1) & 1))) bad = true;
          if (!bad) load_v(i - 1 + kVStages);
        }
      }
    } else if (softmax) {
      for (int i = 0; i < nb; ++i) {
        const long long q = q0 + i;
        const bool tree_blk = blk0 + i == nctx;
        // ---- this thread's 32 scores of the block ----
        if (!bad && !ptx::mbar_wait(&s_bar[q & 1], (uint32_t)((q >> 1) & 1))) bad = true;
        ptx::tc_fence_after();
        float sv[kHalfKeys];
        ptx::tmem_ld32(tq + kColSP + (uint32_t)(q & 1) * kKB + hf * kHalfKeys, sv);
        ptx::tmem_wait_ld();
        // ---- masked, scaled scores and the block maximum of the row ----
        const int key0 = tree_blk ? 0 : (blk0 + i) * kKB;  // key (or node) of column 0
        const int kend = tree_blk ? N : ctx;
        const int kb = key0 + hf * kHalfKeys;  // this half's first key
        float s2[kHalfKeys];
        if (!tree_blk && kb + kHalfKeys <= kend) {
#pragma unroll
          for (int e = 0; e < kHalfKeys; ++e) s2[e] = sv[e] * A.scale_log2;
        } else {
#pragma unroll
          for (int e = 0; e < kHalfKeys; ++e) {
            const bool ok = tree_blk ? ((my_anc >> (kb + e)) & 1ull) != 0 : kb + e < kend;
            s2[e] = ok ? sv[e] * A.scale_log2 : -INFINITY;
          }
        }
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmaxf(s2[e], s2[e + 16]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], mx[e + 8]);
#pragma unroll
        for (int e = 0; e < 4; ++e) mx[e] = fmaxf(mx[e], mx[e + 4]);
        const float mh = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        red[hf * kRows + r] = mh;
        // context keys past the cache's end: their V rows are zeroed, so that a
        // non-finite value there cannot reach O through a zero weight
        const int vrows = kend - key0;
        if (!tree_blk && vrows < kKB && warp == 1) {
          if (!bad && !ptx::mbar_wait(&v_bar[q % kVStages], (uint32_t)((q / kVStages) & 1)))
            bad = true;
          unsigned char *vd = smem + kSmemV + (int)(q % kVStages) * kKBytes;
          const int zr = kKB - vrows;  // rows to clear, in each of the 4 atoms
          for (int idx = lane; idx < (kDh / 64) * zr * 8; idx += 32) {
            const int a = idx / (zr * 8), rm = idx - a * zr * 8;
            *reinterpret_cast<uint4 *>(vd + a * kKVAtom + (vrows + rm / 8) * 128 + (rm % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          ptx::fence_proxy_async();
        }
        ptx::named_sync(1, kSoftmaxThreads);  // ---------------- both halves' maxima
        const float mb = fmaxf(mh, red[(1 - hf) * kRows + r]);
        float alpha = 1.f;
        bool need = false;
        if (mb > m_run + 8.f) {  // move the reference maximum (also the first time)
          alpha = ex2(m_run - mb);
          need = i > 0;  // O holds earlier blocks (of both halves' keys)
          l_run *= alpha;
          m_run = mb;
        }
        // a row with no valid key yet (padding rows) takes 0 as its reference,
        // so that masked keys weigh 2^-inf = 0
        const float mref = m_run == -INFINITY ? 0.f : m_run;
        float p[kHalfKeys];
#pragma unroll
        for (int e = 0; e < kHalfKeys; ++e) p[e] = ex2(s2[e] - mref);
        float sm[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) sm[e] = p[e] + p[e + 16];
#pragma unroll
        for (int e = 0; e < 8; ++e) sm[e] += sm[e + 8];
#pragma unroll
        for (int e = 0; e < 4; ++e) sm[e] += sm[e + 4];
        l_run += (sm[0] + sm[1]) + (sm[2] + sm[3]);
        // rows whose maximum moved rescale their half of O, once the previous
        // P V product is done
        if (__any_sync(0xffffffffu, need)) {
          if (!bad && !ptx::mbar_wait(&o_bar[(q - 1) & 1], (uint32_t)(((q - 1) >> 1) & 1)))
            bad = true;
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHalfCols / 32; ++c) {
            const uint32_t col = tq + kColO + (uint32_t)(hf * kHalfCols + 32 * c);
            float ov[32];
            ptx::tmem_ld32(col, ov);
            ptx::tmem_wait_ld();
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(ov[e] * alpha);
            ptx::tmem_st32(col, w);
          }
        }
        // ---- P (bf16 hi and lo) -> TMEM, over this block's S: every softmax
        // thread has read its scores before the max exchange ----
        ptx::tc_fence_after();
        {
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) split_bf16x2(p[2 * e], p[2 * e + 1], ph[e], pl[e]);
          const uint32_t pc = tq + kColSP + (uint32_t)(q & 1) * kKB + hf * 16;
          ptx::tmem_st16(pc, ph);
          ptx::tmem_st16(pc + kKB / 2, pl);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        mbar_arrive(&p_full[q & 1]);
      }
    }

    // ---- this segment's partial -> workspace (slot (CTA group + KV group)
    // x tiles + tile, unique since along the list either advances by one) ----
    if (softmax && nb > 0 && !bad) {
      const long long ql = q0 + nb - 1;
      if (!ptx::mbar_wait(&o_bar[ql & 1], (uint32_t)((ql >> 1) & 1))) bad = true;
    }
    ptx::tc_fence_after();
    if (softmax) red[hf * kRows + r] = l_run;
    // a wait that timed out anywhere in the CTA ends its work (empty partials
    // from here on, so that every counter still completes)
    if (__syncthreads_or(bad)) aborted = true;
    const bool valid = !aborted;
    float *pp = A.part + (size_t)((cg + kvg) * tiles + tile) * unit_floats(g);
    if (real_row && hf == 0) {
      pp[r] = valid && nb > 0 ? m_run : -INFINITY;
      pp[kRows + r] = valid && nb > 0 ? red[r] + red[kRows + r] : 0.f;
    }
    if (valid && nb > 0 && softmax && quad * 32 < rows) {
      float *orow = pp + 2 * kRows + (size_t)r * kDh + hf * kHalfCols;
#pragma unroll 1
      for (int c = 0; c < kHalfCols / 32; ++c) {
        float ov[32];
        ptx::tmem_ld32(tq + kColO + (uint32_t)(hf * kHalfCols + 32 * c), ov);
        ptx::tmem_wait_ld();
        if (real_row) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(orow + 32 * c + e) =
                make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
        }
      }
    }
    q0 += nb;
    if (bad && A.status) *A.status = LBX_ETIMEOUT;
    __threadfence();
    ptx::tc_fence_before();
    // the row tile's pieces: the CTA groups owning its first and last block
    const long long c_first = owner(g_first), c_last = owner(g_first + nbr - 1);
    if (tid == 0) {
      const unsigned prev = atomicAdd(&A.counters[gidx], 1u);
      misc[1] = (long long)prev == c_last - c_first ? 1 : 0;
    }
    __syncthreads();
    // ---- the last piece of a group merges its partials ----
    if (misc[1]) {
      __threadfence();
      if (real_row) {
        float M = -INFINITY;
        for (long long c = c_first; c <= c_last; ++c) {
          const float *pc = A.part + (size_t)((c + kvg) * tiles + tile) * unit_floats(g);
          M = fmaxf(M, __ldcg(pc + r));
        }
        float Lsum = 0.f;
        for (long long c = c_first; c <= c_last; ++c) {
          const float *pc = A.part + (size_t)((c + kvg) * tiles + tile) * unit_floats(g);
          const float lc = __ldcg(pc + kRows + r);
          if (lc > 0.f) Lsum += exp2f(__ldcg(pc + r) - M) * lc;
        }
        const float inv = 1.f / Lsum;
        const int hl = r / N;
        const int hq = kvh * g.G + h0 + hl;
        float *orow = A.o + (((size_t)lb * N + n_row) * A.Hq + hq) * kDh + hf * kHalfCols;
#pragma unroll 1
        for (int c0 = 0; c0 < kHalfCols; c0 += 32) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
          for (long long c = c_first; c <= c_last; ++c) {
            const float *pc = A.part + (size_t)((c + kvg) * tiles + tile) * unit_floats(g);
            const float lc = __ldcg(pc + kRows + r);
            if (!(lc > 0.f)) continue;
            const float w = exp2f(__ldcg(pc + r) - M);
            const float4 *src = reinterpret_cast<const float4 *>(
                pc + 2 * kRows + (size_t)r * kDh + hf * kHalfCols + c0);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 v = __ldcg(src + e);
              acc[4 * e] = fmaf(w, v.x, acc[4 * e]);
              acc[4 * e + 1] = fmaf(w, v.y, acc[4 * e + 1]);
              acc[4 * e + 2] = fmaf(w, v.z, acc[4 * e + 2]);
              acc[4 * e + 3] = fmaf(w, v.w, acc[4 * e + 3]);
            }
          }
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            __stcs(reinterpret_cast<float4 *>(orow + c0 + e),
                   make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv,
                               acc[e + 3] * inv));
        }
      }
      if (tid == 0) A.counters[gidx] = 0u;  // re-armed for the next call
    }
    __syncthreads();  // red, misc and the Q tile are reused by the next segment
  }

  // ---- drain: copies and MMAs still in flight after an abort ----
  if (issuer && aborted) {
    for (int j = n_kloads - kKStages < 0 ? 0 : n_kloads - kKStages; j < n_kloads; ++j)
      (void)ptx::mbar_wait(&k_bar[j % kKStages], (uint32_t)((j / kKStages) & 1));
    for (int j = n_vloads - kVStages < 0 ? 0 : n_vloads - kVStages; j < n_vloads; ++j)
      (void)ptx::mbar_wait(&v_bar[j % kVStages], (uint32_t)((j / kVStages) & 1));
    if (n_mma1 > 0)
      (void)ptx::mbar_wait(&s_bar[(n_mma1 - 1) & 1], (uint32_t)(((n_mma1 - 1) >> 1) & 1));
    if (n_mma2 > 0)
      (void)ptx::mbar_wait(&o_bar[(n_mma2 - 1) & 1], (uint32_t)(((n_mma2 - 1) >> 1) & 1));
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host side ----------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool have_encode() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// (dh, Hkv, rows) bf16 view of a [rows][Hkv][dh] array; box (64, 1, 32).
bool encode_kv(CUtensorMap *map, const void *base, int Hkv, long long rows) {
  const cuuint64_t gdim[3] = {(cuuint64_t)kDh, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t gstride[2] = {(cuuint64_t)kDh * 2, (cuuint64_t)Hkv * kDh * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kKB};
  const cuuint32_t estride[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), gdim, gstride,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t attn_ws_bytes(int L, int Bq, int N, int Hq, int Hkv, int T) {
  (void)T;
  const Geo g = geometry(L, Bq, N, Hq, Hkv);
  return part_bytes(g) + (((size_t)g.gt * 4 + 255) & ~(size_t)255);
}

bool shapes_ok(int L, int Bq, int N, int Hq, int Hkv, int dh, int T) {
  if (L < 1 || Bq < 1 || N < 1 || N > kMaxNodes || Hq < 1 || Hkv < 1 || T < 0) return false;
  if (dh != kDh || Hq % Hkv != 0) return false;
  if ((long long)L * Bq * T > 0x7fffffffLL || (long long)L * Bq * N * Hq > 0x7fffffffLL)
    return false;
  const Geo g = geometry(L, Bq, N, Hq, Hkv);
  return g.gt <= 0x7fffffffLL;
}

}  // namespace attn
}  // namespace lbx

extern "C" size_t lbx_attn_workspace_size(int L, int Bq, int N, int Hq, int Hkv, int dh, int T) {
  if (!lbx::attn::shapes_ok(L, Bq, N, Hq, Hkv, dh, T)) return 0;
  return lbx::attn::attn_ws_bytes(L, Bq, N, Hq, Hkv, T);
}

extern "C" int lbx_tree_attention(int L, int Bq, int N, int Hq, int Hkv, int dh, int T,
                                  float scale, const int32_t *ctx_len, const int32_t *parent,
                                  const uint16_t *q, const uint16_t *k_cache,
                                  const uint16_t *v_cache, const uint16_t *k_tree,
                                  const uint16_t *v_tree, float *o, void *workspace,
                                  size_t workspace_bytes, int32_t *d_status, cudaStream_t stream) {
  using namespace lbx::attn;
  if (!shapes_ok(L, Bq, N, Hq, Hkv, dh, T)) return LBX_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return LBX_EINVAL;
  auto al = [](const void *p, uintptr_t a) { return p != nullptr && ((uintptr_t)p & (a - 1)) == 0; };
  if (!al(ctx_len, 4) || !al(parent, 4) || !al(q, 16) || !al(k_tree, 16) || !al(v_tree, 16) ||
      !al(o, 16) || !al(workspace, 16) || (d_status && !al(d_status, 4)))
    return LBX_EINVAL;
  if (T > 0 && (!al(k_cache, 16) || !al(v_cache, 16))) return LBX_EINVAL;
  const size_t need = attn_ws_bytes(L, Bq, N, Hq, Hkv, T);
  if (workspace_bytes < need) return LBX_EINVAL;
  if (!have_encode()) return LBX_ECUDA;
  Maps maps;
  std::memset(&maps, 0, sizeof maps);
  if (T > 0 && (!encode_kv(&maps.kc, k_cache, Hkv, (long long)L * Bq * T) ||
                !encode_kv(&maps.vc, v_cache, Hkv, (long long)L * Bq * T)))
    return LBX_ECUDA;
  if (!encode_kv(&maps.kt, k_tree, Hkv, (long long)L * Bq * N) ||
      !encode_kv(&maps.vt, v_tree, Hkv, (long long)L * Bq * N))
    return LBX_ECUDA;
  Args A;
  A.L = L, A.Bq = Bq, A.N = N, A.Hq = Hq, A.Hkv = Hkv, A.T = T;
  A.geo = geometry(L, Bq, N, Hq, Hkv);
  A.scale_log2 = scale * 1.4426950408889634f;
  A.q = q, A.ctx_len = ctx_len, A.parent = parent, A.o = o;
  A.part = static_cast<float *>(workspace);
  A.counters = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(workspace) +
                                                part_bytes(A.geo));
  A.status = d_status;
  if (cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemTotal) != cudaSuccess)
    return LBX_ECUDA;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1)
    return LBX_ECUDA;
  // one CTA per SM, persistent, in groups of `tiles` (at least one group)
  int grid = nsm < kMaxCtas ? nsm : kMaxCtas;
  grid = grid / A.geo.tiles * A.geo.tiles;
  if (grid < A.geo.tiles) grid = A.geo.tiles;
  tree_attn_kernel<<<(unsigned)grid, kThreads, kSmemTotal, stream>>>(maps, A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}
