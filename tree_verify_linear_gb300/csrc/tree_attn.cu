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
// A CTA owns one (layer, request, KV head, row tile, key chunk): row tiles
// hold at most 128 rows (hp heads x N nodes; G x N = 132 at budget 22 with
// 6 heads per KV head gives two tiles of 66), key chunks split the context so
// that the grid fills the GPU, and one extra chunk per row tile holds the
// tree's own keys, with the ancestor mask.  The two row tiles of a chunk are
// adjacent CTAs, so the second read of a K/V block is mostly an L2 hit.
// Each CTA writes its unnormalised partial (running max m, sum l, O) to the
// workspace; the last CTA of a row tile to finish merges the chunks.
//
// Per CTA: the Q tile (128 x 256 bf16, 128-byte swizzled, K-major) stays in
// shared memory; K and V blocks of 32 keys arrive by TMA, four blocks in
// flight; S (two 32-column buffers), P (two buffers, bf16 hi and lo) and O
// (256 columns) live in tensor memory.  P is split into bf16 hi + lo and
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
constexpr int kKStages = 3;             // K blocks in flight (S runs two blocks ahead)
constexpr int kVStages = 2;             // V blocks in flight
constexpr int kMaxNodes = LBX_ATTN_MAX_NODES;
// Target CTA count the context split aims at (four waves of one CTA per SM
// on a 152-SM GPU); a function of the shapes only, so that the workspace
// size does not depend on the device.
constexpr long long kTargetUnits = 608;

// shared memory: Q tile, K stages, V stages, ancestor masks, ints, mbarriers
constexpr int kQBytes = (kDh / 64) * kRows * 128;  // 64 KB, atoms of 64 dh columns
constexpr int kKVAtom = kKB * 128;                 // one 64-column atom of a block
constexpr int kKBytes = (kDh / 64) * kKVAtom;      // 32 KB: one K (or V) block
constexpr int kSmemQ = 0;
constexpr int kSmemK = kQBytes;
constexpr int kSmemV = kSmemK + kKStages * kKBytes;
constexpr int kSmemAnc = kSmemV + kVStages * kKBytes;      // uint64 [64]
constexpr int kSmemRed = kSmemAnc + kMaxNodes * 8;        // float [2][128]
constexpr int kSmemMisc = kSmemRed + 2 * kRows * 4;       // int [16]
constexpr int kSmemBars = kSmemMisc + 64;                 // uint64 [9]
constexpr int kSmemTotal = kSmemBars + 9 * 8;
static_assert(kSmemTotal <= 227 * 1024, "shared memory");
static_assert(kSmemK % 1024 == 0 && kSmemV % 1024 == 0 && kKBytes % 1024 == 0,
              "swizzled operands");
// tensor memory columns
constexpr uint32_t kColS = 0;    // S: two 64-column buffers
constexpr uint32_t kColP = 128;  // P: two buffers of 64 columns (32 hi, 32 lo)
constexpr uint32_t kColO = 256;  // O: 256 columns
constexpr uint32_t kTmemCols = 512;
static_assert(kColO + kDh <= kTmemCols && kColP + 2 * kKB <= kColO, "tensor memory");

// Partition of the work (host and device compute the same).
struct Geo {
  int G;         // query heads per KV head
  int tiles;     // row tiles per (layer, request, KV head)
  int hp;        // heads per row tile (the last may hold fewer)
  int n_chunks;  // context chunks (the tree chunk comes after them)
  int kc;        // keys per context chunk (a multiple of kKB)
  long long gt;  // (layer, request, KV head, tile) groups
  long long units;
  int rows_cap;  // hp * N
};

__host__ __device__ inline Geo geometry(int L, int Bq, int N, int Hq, int Hkv, int T) {
  Geo g;
  g.G = Hq / Hkv;
  g.tiles = 1;
  while (((g.G + g.tiles - 1) / g.tiles) * N > kRows) ++g.tiles;
  g.hp = (g.G + g.tiles - 1) / g.tiles;
  g.tiles = (g.G + g.hp - 1) / g.hp;
  g.gt = (long long)L * Bq * Hkv * g.tiles;
  const int max_blocks = (T + kKB - 1) / kKB;
  long long nc = (kTargetUnits + g.gt - 1) / g.gt - 1;
  if (nc > max_blocks) nc = max_blocks;
  if (nc < 1) nc = 1;
  const int per = (int)((max_blocks + nc - 1) / nc);
  g.kc = (per < 1 ? 1 : per) * kKB;
  g.n_chunks = T > 0 ? (T + g.kc - 1) / g.kc : 0;
  g.units = g.gt * (g.n_chunks + 1);
  g.rows_cap = g.hp * N;
  return g;
}

// Floats of one unit's partial: m[128], l[128], then O rows of 256.
__host__ __device__ inline size_t unit_floats(const Geo &g) {
  return 2 * (size_t)kRows + (size_t)g.rows_cap * kDh;
}
__host__ __device__ inline size_t part_bytes(const Geo &g) {
  return ((size_t)g.units * unit_floats(g) * 4 + 255) & ~(size_t)255;
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

__global__ void __launch_bounds__(2 * kRows, 1)
    tree_attn_kernel(const __grid_constant__ Maps maps, const Args A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Geo &g = A.geo;
  const int N = A.N;
  int *misc = reinterpret_cast<int *>(smem + kSmemMisc);  // [0] TMEM base, [1] last CTA
  uint64_t *anc = reinterpret_cast<uint64_t *>(smem + kSmemAnc);
  float *red = reinterpret_cast<float *>(smem + kSmemRed);  // [2][kRows] per-half values
  uint64_t *k_bar = reinterpret_cast<uint64_t *>(smem + kSmemBars);  // [3]
  uint64_t *v_bar = k_bar + 3;                                        // [2]
  uint64_t *s_bar = k_bar + 5;                                        // [2]
  uint64_t *o_bar = k_bar + 7;                                        // [2]

  // ---- the unit: (l*Bq + b, KV head, chunk, tile), tile fastest ----
  long long u = blockIdx.x;
  const int tile = (int)(u % g.tiles);
  u /= g.tiles;
  const int chunk = (int)(u % (g.n_chunks + 1));
  u /= g.n_chunks + 1;
  const int kvh = (int)(u % A.Hkv);
  const int lb = (int)(u / A.Hkv);
  const int b = lb % A.Bq;
  const long long gidx = (long long)lb * A.Hkv * g.tiles + (long long)kvh * g.tiles + tile;
  const bool tree_unit = chunk == g.n_chunks;
  const int h0 = tile * g.hp;
  const int hp_t = g.G - h0 < g.hp ? g.G - h0 : g.hp;
  const int rows = hp_t * N;

  // ---- whole-batch validation (the same verdict in every CTA) ----
  {
    int bad_in = 0;
    for (int i = tid; i < A.Bq * N; i += 2 * kRows) {
      const int n = i % N, p = A.parent[i];
      if (n == 0 ? p != -1 : (p < 0 || p >= n)) bad_in = 1;
    }
    for (int i = tid; i < A.Bq; i += 2 * kRows)
      if (A.ctx_len[i] < 0 || A.ctx_len[i] > A.T) bad_in = 1;
    if (__syncthreads_or(bad_in)) {
      if (tid == 0 && A.status) *A.status = LBX_ETREE;
      return;
    }
  }
  const int ctx = A.ctx_len[b];
  // blocks of this unit, first key, end of the existing keys
  int nb, key0, kend;
  if (tree_unit) {
    nb = (N + kKB - 1) / kKB;
    key0 = 0;
    kend = N;
  } else {
    key0 = chunk * g.kc;
    kend = ctx < key0 + g.kc ? ctx : key0 + g.kc;
    nb = kend > key0 ? (kend - key0 + kKB - 1) / kKB : 0;
  }

  // ---- set-up ----
  if (tid == 0) {
    for (int i = 0; i < 9; ++i) ptx::mbar_init(k_bar + i, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t *>(&misc[0]), kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  if (tree_unit && tid < N) {  // ancestor-or-self mask of node tid
    uint64_t m = 0;
    int j = tid;
    for (int s = 0; s < kMaxNodes && j >= 0; ++s) {
      m |= 1ull << j;
      j = A.parent[(size_t)b * N + j];
    }
    anc[tid] = m;
  }
  // Q tile: row r = hl * N + n (head hl of the tile, node n), zero padding rows
  {
    const uint4 *qg = reinterpret_cast<const uint4 *>(A.q);
    for (int idx = tid; idx < kRows * (kDh / 8); idx += 2 * kRows) {
      const int r = idx / (kDh / 8), c16 = idx % (kDh / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const int hl = r / N, n = r - hl * N;
        const int hq = kvh * g.G + h0 + hl;
        v = qg[(((size_t)lb * N + n) * A.Hq + hq) * (kDh / 8) + c16];
      }
      const int atom = c16 >> 3, ch = c16 & 7;
      *reinterpret_cast<uint4 *>(smem + kSmemQ + atom * (kRows * 128) + r * 128 +
                                 ((ch ^ (r & 7)) << 4)) = v;
    }
  }
  ptx::fence_proxy_async();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int quad = warp & 3, hf = warp >> 2;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);  // this warp's lane quadrant

  const int r = quad * 32 + lane;
  const bool real_row = r < rows;
  const int n_row = real_row ? r - (r / N) * N : 0;
  // tree unit: the ancestor bits of this thread's 16 keys of each block
  const uint64_t my_anc = tree_unit && real_row ? anc[n_row] : 0ull;

  const bool lead = tid == 0;
  int n_kloads = 0, n_vloads = 0, n_mma1 = 0, n_mma2 = 0;  // issued by the lead
  const int zbase = tree_unit ? lb * N : lb * A.T + key0;  // position row of block 0
  const CUtensorMap *mk = tree_unit ? &maps.kt : &maps.kc;
  const CUtensorMap *mv = tree_unit ? &maps.vt : &maps.vc;
  auto load_k = [&](int j) {
    const int s = j % kKStages;
    unsigned char *kd = smem + kSmemK + s * kKBytes;
    ptx::mbar_arrive_expect_tx(&k_bar[s], (uint32_t)kKBytes);
#pragma unroll
    for (int a = 0; a < kDh / 64; ++a)
      ptx::tma_load_3d(kd + a * kKVAtom, mk, a * 64, kvh, zbase + j * kKB, &k_bar[s]);
    ++n_kloads;
  };
  auto load_v = [&](int j) {
    const int s = j % kVStages;
    unsigned char *vd = smem + kSmemV + s * kKBytes;
    ptx::mbar_arrive_expect_tx(&v_bar[s], (uint32_t)kKBytes);
#pragma unroll
    for (int a = 0; a < kDh / 64; ++a)
      ptx::tma_load_3d(vd + a * kKVAtom, mv, a * 64, kvh, zbase + j * kKB, &v_bar[s]);
    ++n_vloads;
  };
  // descriptors of the Q tile and of stage 0; the others are fixed offsets
  // (added to the 16-byte address field)
  const uint64_t qdesc = ptx::sdesc_sw128(ptx::smem_u32(smem + kSmemQ));
  const uint64_t kdesc0 = ptx::sdesc_sw128(ptx::smem_u32(smem + kSmemK));
  const uint64_t vdesc0 =
      ptx::sdesc(ptx::smem_u32(smem + kSmemV), (uint32_t)kKVAtom, 1024u, 2u);
  // S[j & 1] = Q K_j^T: M = 128, N = 64 keys, K = 256 (16 steps)
  auto mma1 = [&](int j) {
    const uint64_t kd = kdesc0 + (uint64_t)(((j % kKStages) * kKBytes) >> 4);
    constexpr uint32_t idesc = ptx::idesc_bf16(128, kKB);
    const uint32_t d = tmem + kColS + (uint32_t)(j & 1) * kKB;
#pragma unroll
    for (int ks = 0; ks < kDh / 16; ++ks) {
      const uint64_t ao = (uint64_t)(((ks >> 2) * (kRows * 128) + (ks & 3) * 32) >> 4);
      const uint64_t bo = (uint64_t)(((ks >> 2) * kKVAtom + (ks & 3) * 32) >> 4);
      ptx::mma_bf16_ss(d, qdesc + ao, kd + bo, idesc, ks > 0 ? 1u : 0u);
    }
    ptx::mma_commit(&s_bar[j & 1]);
    ++n_mma1;
  };
  // O += P_j V_j: A = P (TMEM, hi then lo), B = the V block read MN-major
  // (dh contiguous in 64-column atoms kKVAtom apart, 8-key groups 1024 apart)
  auto mma2 = [&](int j, bool acc) {
    const uint64_t vd = vdesc0 + (uint64_t)(((j % kVStages) * kKBytes) >> 4);
    constexpr uint32_t idesc = ptx::idesc_bf16_bmn(128, kDh);
    const uint32_t pc = tmem + kColP + (uint32_t)(j & 1) * kKB;
    uint32_t accum = acc ? 1u : 0u;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass)
#pragma unroll
      for (int ks = 0; ks < kKB / 16; ++ks) {
        ptx::mma_bf16_ts(tmem + kColO, pc + pass * (kKB / 2) + ks * 8,
                         vd + (uint64_t)(ks * 2048 >> 4), idesc, accum);
        accum = 1u;
      }
    ptx::mma_commit(&o_bar[j & 1]);
    ++n_mma2;
  };

  bool bad = false, aborted = false;
  if (lead && nb > 0) {
    for (int j = 0; j < nb && j < kKStages; ++j) load_k(j);
    for (int j = 0; j < nb && j < kVStages; ++j) load_v(j);
    if (!ptx::mbar_wait(&k_bar[0], 0u)) bad = true;
    mma1(0);
  }

  float m_run = -INFINITY, l_run = 0.f;  // base-2 running max; this half's sum
  for (int i = 0; i < nb; ++i) {
    // ---- this thread's 16 scores of block i ----
    if (!ptx::mbar_wait(&s_bar[i & 1], (uint32_t)((i >> 1) & 1))) bad = true;
    ptx::tc_fence_after();
    float sv[kHalfKeys];
    ptx::tmem_ld32(tq + kColS + (uint32_t)(i & 1) * kKB + hf * kHalfKeys, sv);
    ptx::tmem_wait_ld();
    if (lead) {
      // K_i has been read (S_i is complete): its stage takes block i + 3
      if (i + kKStages < nb) load_k(i + kKStages);
      // the next block's scores, into the other buffer (read in iteration i-1)
      if (i + 1 < nb) {
        if (!ptx::mbar_wait(&k_bar[(i + 1) % kKStages], (uint32_t)(((i + 1) / kKStages) & 1)))
          bad = true;
        mma1(i + 1);
      }
    }
    // ---- masked, scaled scores and the block maximum of the row ----
    const int kb = key0 + i * kKB + hf * kHalfKeys;  // this half's first key
    float s2[kHalfKeys];
    if (!tree_unit && kb + kHalfKeys <= kend) {
#pragma unroll
      for (int e = 0; e < kHalfKeys; ++e) s2[e] = sv[e] * A.scale_log2;
    } else {
#pragma unroll
      for (int e = 0; e < kHalfKeys; ++e) {
        const bool ok = tree_unit ? ((my_anc >> (kb + e)) & 1ull) != 0 : kb + e < kend;
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
    float mh = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    red[hf * kRows + r] = mh;
    // context keys past the cache's end: their V rows are zeroed, so that a
    // non-finite value there cannot reach O through a zero weight
    const int vrows = kend - (key0 + i * kKB);
    if (!tree_unit && vrows < kKB && warp == 1) {
      if (!ptx::mbar_wait(&v_bar[i % kVStages], (uint32_t)((i / kVStages) & 1))) bad = true;
      unsigned char *vd = smem + kSmemV + (i % kVStages) * kKBytes;
      const int zr = kKB - vrows;  // rows to clear, in each of the 4 atoms
      for (int idx = lane; idx < (kDh / 64) * zr * 8; idx += 32) {
        const int a = idx / (zr * 8), rem = idx - a * zr * 8;
        *reinterpret_cast<uint4 *>(vd + a * kKVAtom + (vrows + rem / 8) * 128 + (rem % 8) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      ptx::fence_proxy_async();
    }
    __syncthreads();  // ---------------------------------------------- both halves' maxima
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
    // rows whose maximum moved rescale their half of O, once MMA2_{i-1} is done
    if (__any_sync(0xffffffffu, need)) {
      if (!ptx::mbar_wait(&o_bar[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1))) bad = true;
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
    // ---- P_i (bf16 hi and lo) -> TMEM ----
    {
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) split_bf16x2(p[2 * e], p[2 * e + 1], ph[e], pl[e]);
      const uint32_t pc = tq + kColP + (uint32_t)(i & 1) * kKB + hf * 16;
      ptx::tmem_st16(pc, ph);
      ptx::tmem_st16(pc + kKB / 2, pl);
    }
    // the lead: MMA2_{i-1} complete (O, its P buffer and its V stage free),
    // then block i + 1's values into that stage
    if (lead && i >= 1) {
      if (!ptx::mbar_wait(&o_bar[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1))) bad = true;
      if (i + 1 < nb) load_v(i + 1);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    if (__syncthreads_or(bad)) {  // ------------------------------------ P_i complete
      aborted = true;
      break;
    }
    if (lead) {
      if (!ptx::mbar_wait(&v_bar[i % kVStages], (uint32_t)((i / kVStages) & 1))) bad = true;
      ptx::tc_fence_after();
      mma2(i, i > 0);
    }
  }

  // ---- partial of this unit -> workspace ----
  if (!aborted && nb > 0) {
    if (!ptx::mbar_wait(&o_bar[(nb - 1) & 1], (uint32_t)(((nb - 1) >> 1) & 1))) bad = true;
  }
  ptx::tc_fence_after();
  red[hf * kRows + r] = l_run;
  __syncthreads();
  const bool valid = !aborted && !bad;
  float *pp = A.part + (size_t)blockIdx.x * unit_floats(g);
  if (real_row && hf == 0) {
    pp[r] = valid ? m_run : -INFINITY;
    pp[kRows + r] = valid ? red[r] + red[kRows + r] : 0.f;
  }
  if (valid && nb > 0 && quad * 32 < rows) {
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
  if (bad && A.status) *A.status = LBX_ETIMEOUT;
  __threadfence();
  ptx::tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&A.counters[gidx], 1u);
    misc[1] = prev == (unsigned)g.n_chunks ? 1 : 0;  // n_chunks + 1 units per group
  }
  // drain: copies and MMAs still in flight after an abort
  if (lead && aborted) {
    for (int j = n_kloads - kKStages < 0 ? 0 : n_kloads - kKStages; j < n_kloads; ++j)
      (void)ptx::mbar_wait(&k_bar[j % kKStages], (uint32_t)((j / kKStages) & 1));
    for (int j = n_vloads - kVStages < 0 ? 0 : n_vloads - kVStages; j < n_vloads; ++j)
      (void)ptx::mbar_wait(&v_bar[j % kVStages], (uint32_t)((j / kVStages) & 1));
    if (n_mma1 > 0)
      (void)ptx::mbar_wait(&s_bar[(n_mma1 - 1) & 1], (uint32_t)(((n_mma1 - 1) >> 1) & 1));
    if (n_mma2 > 0)
      (void)ptx::mbar_wait(&o_bar[(n_mma2 - 1) & 1], (uint32_t)(((n_mma2 - 1) >> 1) & 1));
  }
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }

  // ---- the last unit of a row tile merges the chunks ----
  if (misc[1]) {
    __threadfence();
    if (real_row) {
      const long long first = (long long)blockIdx.x - (long long)chunk * g.tiles;
      float M = -INFINITY;
      for (int c = 0; c <= g.n_chunks; ++c) {
        const float *pc = A.part + (size_t)(first + (long long)c * g.tiles) * unit_floats(g);
        M = fmaxf(M, __ldcg(pc + r));
      }
      float Lsum = 0.f;
      for (int c = 0; c <= g.n_chunks; ++c) {
        const float *pc = A.part + (size_t)(first + (long long)c * g.tiles) * unit_floats(g);
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
        for (int c = 0; c <= g.n_chunks; ++c) {
          const float *pc = A.part + (size_t)(first + (long long)c * g.tiles) * unit_floats(g);
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
                 make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv));
      }
    }
    if (tid == 0) A.counters[gidx] = 0u;  // re-armed for the next call
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
  const Geo g = geometry(L, Bq, N, Hq, Hkv, T);
  return part_bytes(g) + (((size_t)g.gt * 4 + 255) & ~(size_t)255);
}

bool shapes_ok(int L, int Bq, int N, int Hq, int Hkv, int dh, int T) {
  if (L < 1 || Bq < 1 || N < 1 || N > kMaxNodes || Hq < 1 || Hkv < 1 || T < 0) return false;
  if (dh != kDh || Hq % Hkv != 0) return false;
  if ((long long)L * Bq * T > 0x7fffffffLL || (long long)L * Bq * N * Hq > 0x7fffffffLL)
    return false;
  const Geo g = geometry(L, Bq, N, Hq, Hkv, T);
  return g.units <= 0x7fffffffLL;
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
  A.geo = geometry(L, Bq, N, Hq, Hkv, T);
  A.scale_log2 = scale * 1.4426950408889634f;
  A.q = q, A.ctx_len = ctx_len, A.parent = parent, A.o = o;
  A.part = static_cast<float *>(workspace);
  A.counters = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(workspace) +
                                                part_bytes(A.geo));
  A.status = d_status;
  if (cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemTotal) != cudaSuccess)
    return LBX_ECUDA;
  tree_attn_kernel<<<(unsigned)A.geo.units, 2 * kRows, kSmemTotal, stream>>>(maps, A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}
