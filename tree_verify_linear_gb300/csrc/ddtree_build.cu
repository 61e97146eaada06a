// ddtree_build.cu -- DDTree construction from the draft's top-K scores, on
// the device.
//
// Lucebox hub README: DDTree is the tree-structured verify that beats chain
// verify at the same budget ("Algorithms used"), budget 22 on the RTX 3090
// ("Implemented here"), and the draft's top-K tokens per position come from a
// device kernel ("GPU draft top-K & verify-argmax (DFlash)").  The tree of
// budget B is built best first: a node's score is the sum (fp32, from the
// root down) of the draft log-probabilities along its path; starting from the
// root, the not-yet-added child of an added node with the highest score joins
// next (ties: the lower parent, then the lower k), until B nodes or no
// candidate is left.  Nodes are numbered in the order they join, so the
// parent array is topologically numbered and feeds lbx_verify_step as is.
//
// One warp per request.  The candidates -- every child (u, k) of every added
// node -- sit in shared memory in the order they are created, which is (u, k)
// order, so "lowest candidate index" is the tie rule; each round the warp
// finds the best unused candidate with a shuffle reduction, appends the new
// node and its K children.
#include <math.h>
#include <stdint.h>

#include "lbx.h"

namespace lbx {
namespace {

constexpr int kDtWarps = 4;  // requests per CTA
constexpr int kDtMaxCand = LBX_MAX_TREE_NODES * LBX_DDTREE_MAX_K;

struct DtArgs {
  int Bq, D, K, B;
  const float *logp;
  const int32_t *tok, *root_tok;
  int32_t *parent, *token, *depth, *n_nodes;
  float *score;
};

__global__ void __launch_bounds__(32 * kDtWarps) ddtree_build_kernel(const DtArgs A) {
  __shared__ float c_s[kDtWarps][kDtMaxCand];  // candidate score
  __shared__ int c_u[kDtWarps][kDtMaxCand];    // candidate parent (-1: taken)
  __shared__ int c_k[kDtWarps][kDtMaxCand];    // candidate slot k
  __shared__ int n_d[kDtWarps][LBX_MAX_TREE_NODES];
  __shared__ float t_lp[kDtWarps][LBX_DDTREE_MAX_DEPTH * LBX_DDTREE_MAX_K];  // the request's
  __shared__ int t_tk[kDtWarps][LBX_DDTREE_MAX_DEPTH * LBX_DDTREE_MAX_K];    // top-K table
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * kDtWarps + w;
  if (b >= A.Bq) return;
  const int D = A.D, K = A.K, B = A.B;
  // the request's top-K table, staged once (every round reads it)
  float *lp = t_lp[w];
  int *tk = t_tk[w];
  for (int i = lane; i < D * K; i += 32) {
    lp[i] = A.logp[(size_t)b * D * K + i];
    tk[i] = A.tok[(size_t)b * D * K + i];
  }
  __syncwarp();
  int32_t *par = A.parent + (size_t)b * B, *tn = A.token + (size_t)b * B;
  int32_t *dep = A.depth ? A.depth + (size_t)b * B : nullptr;
  float *sco = A.score ? A.score + (size_t)b * B : nullptr;
  for (int i = lane; i < B; i += 32) {
    par[i] = -1;
    tn[i] = i == 0 ? A.root_tok[b] : -1;
    if (dep) dep[i] = i == 0 ? 0 : -1;
    if (sco) sco[i] = 0.f;
  }
  float *cs = c_s[w];
  int *cu = c_u[w], *ck = c_k[w], *nd = n_d[w];
  if (lane == 0) nd[0] = 0;
  int cnt = 0;
  if (D > 0) {
    if (lane < K) cs[lane] = 0.f + lp[lane], cu[lane] = 0, ck[lane] = lane;
    cnt = K;
  }
  __syncwarp();
  int n = 1;
  for (; n < B; ++n) {
    // best unused candidate: highest score, then lowest index
    float bs = 0.f;
    int bi = -1;
    for (int c = lane; c < cnt; c += 32)
      if (cu[c] >= 0 && (bi < 0 || cs[c] > bs)) bs = cs[c], bi = c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi >= 0 && (bi < 0 || os > bs || (os == bs && oi < bi))) bs = os, bi = oi;
    }
    if (bi < 0) break;  // the whole trie is in
    const int u = cu[bi], k = ck[bi], du = nd[u];
    __syncwarp();  // every lane has read the candidate before it is marked
    if (lane == 0) {
      cu[bi] = -1;
      nd[n] = du + 1;
      par[n] = u;
      tn[n] = tk[du * K + k];
      if (dep) dep[n] = du + 1;
      if (sco) sco[n] = bs;
    }
    // the new node's children
    if (du + 1 < D) {
      if (lane < K) {
        cs[cnt + lane] = bs + lp[(du + 1) * K + lane];
        cu[cnt + lane] = n;
        ck[cnt + lane] = lane;
      }
      cnt += K;
    }
    __syncwarp();
  }
  if (lane == 0) A.n_nodes[b] = n;
}

}  // namespace
}  // namespace lbx

extern "C" int lbx_ddtree_build(int Bq, int D, int K, int B, const float *logp,
                                const int32_t *tok, const int32_t *root_tok, int32_t *parent_out,
                                int32_t *token_out, int32_t *depth_out, float *score_out,
                                int32_t *n_nodes_out, cudaStream_t stream) {
  if (Bq < 1 || D < 0 || D > LBX_DDTREE_MAX_DEPTH || K < 1 || K > LBX_DDTREE_MAX_K || B < 1 ||
      B > LBX_MAX_TREE_NODES)
    return LBX_EINVAL;
  auto ok4 = [](const void *p) { return p != nullptr && ((uintptr_t)p & 3u) == 0; };
  if ((D > 0 && (!ok4(logp) || !ok4(tok))) || !ok4(root_tok) || !ok4(parent_out) ||
      !ok4(token_out) || !ok4(n_nodes_out) || (depth_out && !ok4(depth_out)) ||
      (score_out && !ok4(score_out)))
    return LBX_EINVAL;
  lbx::DtArgs A;
  A.Bq = Bq, A.D = D, A.K = K, A.B = B;
  A.logp = logp, A.tok = tok, A.root_tok = root_tok;
  A.parent = parent_out, A.token = token_out, A.depth = depth_out, A.score = score_out;
  A.n_nodes = n_nodes_out;
  const int grid = (Bq + lbx::kDtWarps - 1) / lbx::kDtWarps;
  lbx::ddtree_build_kernel<<<grid, 32 * lbx::kDtWarps, 0, stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? LBX_OK : LBX_ECUDA;
}
