/*
 * lbx.h -- C ABI of the tree-verify gated-DeltaNet library (GB300, sm_103a).
 *
 * The library computes the verify step of a hybrid model's gated-DeltaNet
 * (linear-attention) layers for a DDTree draft tree: the three tree-aware
 * state-rollback operations named in the Lucebox hub README (section
 * "02 DFlash DDtree", list "Implemented here": ggml_ssm_conv_tree,
 * ggml_gated_delta_net_tree, ggml_gated_delta_net_tree_persist), plus one
 * fused entry point that performs all three in a single pass.  DDTree itself
 * (same section, "Algorithms used") is a tree-structured verify: the draft is
 * a tree of B nodes given as a parent-index array, and every node is verified
 * against the state reached along its own root-to-node path.
 *
 * Notation.  L layers, Bq requests, N tree nodes (the budget), Hk key heads,
 * Hv value heads (Hv % Hk == 0; value head h reads key head h / (Hv/Hk)),
 * d = d_k = d_v, K conv width, C = 2*Hk*d + Hv*d conv channels ordered
 * q | k | v.  For each layer, request and value head h the recurrence is the
 * gated delta rule
 *     S_n = a_n S_p (I - b_n k_n k_n^T) + b_n v_n k_n^T,   o_n = q_scale * S_n q_n,
 * where p = parent[n] and S_p of the root (node 0) is the cached state of the
 * request's slot.  S is d_v x d_k, stored row-major [d_v][d_k].
 *
 * Conventions shared by every entry point:
 *   - Every array pointer is a DEVICE pointer owned by the caller; the
 *     library allocates nothing.  bf16 values are passed as their 16-bit
 *     patterns (uint16_t).  All arrays are dense and row-major in the index
 *     order written next to them; each must be 16-byte aligned.
 *   - Calls are asynchronous on `stream`.  The return value reports host-side
 *     argument checks and the launch: LBX_OK, LBX_EINVAL or LBX_ECUDA.
 *   - Structural errors that only the device can see (a parent array that is
 *     not a topologically numbered tree, a slot or accepted index out of
 *     range, two requests naming the same slot, a chain-mode input that is
 *     not a chain) are reported through `d_status` (an int32 in device memory,
 *     may be NULL): the kernel stores LBX_ETREE or LBX_EINVAL there and then
 *     writes NOTHING -- no outputs, no cache update.  `d_status` is never
 *     cleared by the library; zero it before the call to read it afterwards.
 *   - The draft tree: parent[b][0] == -1 (node 0 is the root, the last
 *     accepted token), and 0 <= parent[b][i] < i for i > 0.  One tree per
 *     request is shared by all layers.
 *   - Caches: state[L][n_slots][Hv][d][d] fp32 and conv_cache[L][n_slots][K-1][C]
 *     fp32 (raw pre-conv inputs, oldest row first; with K == 1 there is no
 *     conv cache and its pointer may be NULL).  Request b uses slot
 *     slot[b]; slots that no request names are never read or written.
 */
#ifndef LBX_H
#define LBX_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define LBX_OK 0
#define LBX_EINVAL (-1) /* bad dimension, NULL pointer, size over a limit   */
#define LBX_ECUDA (-2)  /* a CUDA call or kernel launch failed               */
#define LBX_ETREE (-3)  /* invalid tree (device-detected, via d_status)      */
#define LBX_ETIMEOUT (-4) /* a bounded in-kernel wait gave up (via d_status) */

/* Limits. */
#define LBX_MAX_TREE_NODES 64 /* tree mode: N <= 64 nodes per request          */
#define LBX_CHAIN_CHUNK 64    /* chunked mode, CUDA-core path (d != 128): tokens
                                 per chunk; the d = 128 tensor-core chain kernel
                                 walks the chain 16 tokens at a time           */
#define LBX_MAX_CONV_WIDTH 4  /* 1 <= K <= 4                                    */
#define LBX_ACCEPT_MAX_NODES 4096 /* lbx_accept_walk: N <= 4096 nodes         */
#define LBX_DDTREE_MAX_K 8        /* lbx_ddtree_build: top-K, 1 <= K <= 8       */
#define LBX_DDTREE_MAX_DEPTH 64   /* lbx_ddtree_build: draft positions D <= 64  */
#define LBX_ATTN_HEAD_DIM 256     /* lbx_tree_attention: head dimension         */
#define LBX_ATTN_MAX_NODES 64     /* lbx_tree_attention: N <= 64 tree nodes     */

/* Modes of lbx_verify_step. */
#define LBX_MODE_AUTO 0    /* tree if N <= LBX_MAX_TREE_NODES, else chunked     */
#define LBX_MODE_TREE 1    /* arbitrary tree, N <= LBX_MAX_TREE_NODES           */
#define LBX_MODE_CHUNKED 2 /* chain only (parent[i] == i-1), any N >= 1         */
#define LBX_MODE_TREE_CUDA_CORES 3 /* tree mode forced onto the CUDA-core kernel
                                      (same results; for cross-checking)       */

typedef struct lbx_cfg {
  int L;       /* gated-DeltaNet layers in the call (>= 1)                     */
  int Bq;      /* requests (>= 1)                                              */
  int N;       /* tree nodes per request (>= 1)                                */
  int Hk, Hv;  /* key / value heads, Hv % Hk == 0                              */
  int d;       /* head dimension d_k = d_v; 32 or 128                          */
  int K;       /* conv width, 1..LBX_MAX_CONV_WIDTH                            */
  int n_slots; /* cache slots in state / conv_cache (>= Bq)                    */
  float l2_eps;  /* q, k <- x / sqrt(sum x^2 + l2_eps); typical 1e-6           */
  float q_scale; /* o_n = q_scale * S_n q_n; 1.0 for the plain recurrence      */
  int mode;      /* LBX_MODE_*; used by lbx_verify_step only                   */
} lbx_cfg;

/* Human-readable text for a status code (static storage). */
const char *lbx_strerror(int status);

/* Bytes of workspace lbx_verify_step needs for cfg (0 on a bad cfg).  It
 * must be zero-filled once before its first use; two calls that run at the
 * same time must not share a workspace.  What it holds depends on the kernel
 * the configuration selects:
 *   - the tensor-core step (tree mode, d = 128, N <= 64): the per-request
 *     tree tables, per-(layer, request, key head) q/k operands (24 KB each
 *     at N <= 24, 64 KB at N <= 64) and per-(layer, request, value head)
 *     T/W records (2.8 KB at N <= 24, 17 KB at N <= 64) that its prep kernel
 *     writes and its step kernel reads, rewritten by every call;
 *   - the CUDA-core kernels: one arrival counter per (layer, request, key
 *     head); every call that runs to completion leaves them zero again. */
size_t lbx_workspace_size(const lbx_cfg *cfg);

/*
 * Tree conv (ggml_ssm_conv_tree; Lucebox hub README, "02 DFlash DDtree").
 * For node n and channel c:
 *     y = sum_{j=0}^{K-1} conv_w[l][c][K-1-j] * xhat_j[c],   out = y * sigmoid(y)
 * where xhat_0 is node n's input, xhat_1 its parent's, and so on up the
 * ancestor path; past the root the window continues into the slot's conv
 * cache, most recent cached row first.  Then q and k are L2-normalised per
 * key head over d channels (v is not).
 *   x          [L][Bq][N][C]   bf16   raw inputs of the tree nodes
 *   conv_w     [L][C][K]       bf16   depthwise conv weights, no bias
 *   conv_cache [L][n_slots][K-1][C] fp32 (read only here)
 *   parent     [Bq][N] int32, slot [Bq] int32
 *   qkv_out    [L][Bq][N][C]   fp32   (q scaled by nothing; q_scale is applied
 *                                      by lbx_tree_deltanet)
 * Requires cfg->N <= LBX_MAX_TREE_NODES.
 */
int lbx_tree_conv(const lbx_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                  const float *conv_cache, const int32_t *parent, const int32_t *slot,
                  float *qkv_out, int32_t *d_status, cudaStream_t stream);

/*
 * Tree gated delta-rule recurrence (ggml_gated_delta_net_tree; same page).
 * Every node's state is the recurrence along its root-to-node path, started
 * from state[l][slot[b]][h]; o_n = q_scale * S_n q_n.
 *   qkv         [L][Bq][N][C]          fp32 (output of lbx_tree_conv)
 *   a, b        [L][Bq][N][Hv]         bf16 gates, already activated
 *   state       [L][n_slots][Hv][d][d] fp32 (read only here)
 *   parent      [Bq][N], slot [Bq]     int32
 *   o           [L][Bq][N][Hv][d]      fp32
 *   node_states [L][Bq][N][Hv][d][d]   fp32 per-node snapshots for a later
 *                                      lbx_tree_persist; may be NULL
 * Requires cfg->N <= LBX_MAX_TREE_NODES.
 */
int lbx_tree_deltanet(const lbx_cfg *cfg, const float *qkv, const uint16_t *a, const uint16_t *b,
                      const float *state, const int32_t *parent, const int32_t *slot, float *o,
                      float *node_states, int32_t *d_status, cudaStream_t stream);

/*
 * Persist (ggml_gated_delta_net_tree_persist; same page, "state rollback").
 * For each layer l and request b, with acc = accepted[b]:
 *   state[l][slot[b]]      <- node_states[l][b][acc]          (all Hv heads)
 *   conv_cache[l][slot[b]] <- the last K-1 entries of
 *                             [old cache rows, x of the path root..acc]
 * Both caches are updated in place.  The conv part copies bf16-exact values
 * and is bit-exact.
 *   x           [L][Bq][N][C] bf16, node_states [L][Bq][N][Hv][d][d] fp32,
 *   parent [Bq][N], slot [Bq], accepted [Bq] int32.
 */
int lbx_tree_persist(const lbx_cfg *cfg, const uint16_t *x, const float *node_states,
                     const int32_t *parent, const int32_t *slot, const int32_t *accepted,
                     float *state, float *conv_cache, int32_t *d_status, cudaStream_t stream);

/*
 * Fused verify step: tree conv + tree recurrence + persist in one pass.  The
 * cached state is read once, per-node states are never materialised, o is
 * written for every node, and only the accepted node's state and conv window
 * are written back (in place) to each request's slot.
 *   x [L][Bq][N][C], conv_w [L][C][K], a, b [L][Bq][N][Hv]   bf16
 *   parent [Bq][N], slot [Bq], accepted [Bq]                 int32
 *   state [L][n_slots][Hv][d][d], conv_cache [L][n_slots][K-1][C]  fp32, in/out
 *   o [L][Bq][N][Hv][d]                                     fp32, out
 *   workspace / workspace_bytes: >= lbx_workspace_size(cfg) bytes (see there)
 * Modes: in tree mode N <= LBX_MAX_TREE_NODES (the tensor-core step keeps node
 * labels as bytes, two nodes per lane of the warp that builds a request's
 * tables, and the CUDA-core step's S0 [K|Q] product tile covers at most 2N =
 * 128 columns at d = 128); chunked mode takes a chain of any length: at d =
 * 128 on the tensor cores in chunks of 16 tokens, otherwise on CUDA cores in
 * chunks of LBX_CHAIN_CHUNK tokens.  Distinct requests must name distinct
 * slots.
 */
int lbx_verify_step(const lbx_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                    const uint16_t *a, const uint16_t *b, const int32_t *parent,
                    const int32_t *slot, const int32_t *accepted, float *state, float *conv_cache,
                    float *o, void *workspace, size_t workspace_bytes, int32_t *d_status,
                    cudaStream_t stream);

/* Capacity of lbx_verify_step_noalloc: L * Bq * Hk <= LBX_NOALLOC_MAX_GROUPS
 * arrival counters (256 KB). */
#define LBX_NOALLOC_MAX_GROUPS 65536

/*
 * lbx_verify_step without a workspace, for callers that cannot allocate
 * device memory -- for instance an engine that reserves all device memory
 * for its caches up front and allows no later cudaMalloc (which would also
 * synchronise the device), or a plugin inside a host framework that owns the
 * only allocator.  It computes exactly what lbx_verify_step computes; the
 * Lucebox hub README describes no such variant, so it has no passage of its
 * own to cite.
 *
 * Arguments and results are those of lbx_verify_step minus the workspace.
 * The arrival counters live in a fixed device array inside the library
 * (LBX_NOALLOC_MAX_GROUPS counters, 256 KB), which every GPU that loads the
 * library keeps until the process exits.  Configurations with
 * L * Bq * Hk > LBX_NOALLOC_MAX_GROUPS are rejected with LBX_EINVAL.  Where
 * lbx_verify_step would run the tensor-core step, whose workspace is larger
 * than the array, this function runs the CUDA-core tree kernel instead
 * (results agree within the tolerances of the tests; only speed differs).
 * The function allocates nothing: no cudaMalloc, cudaFree or other
 * allocating call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and may be the moment
 *     the library's kernels and the array are loaded onto that device; make
 *     that first call during set-up, before any stream capture.  The address
 *     is kept for the life of the process: it does not survive
 *     cudaDeviceReset (or any other teardown of the device's primary
 *     context), after which this entry point must not be called again.
 *   - Each call clears the counters it uses (cudaMemsetAsync on `stream`)
 *     before launching, since the array keeps the previous call's contents.
 *   - All calls on a device share the one array: calls that overlap on the
 *     GPU (other streams, other host threads) race on it.  Serialise them.
 */
int lbx_verify_step_noalloc(const lbx_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                            const uint16_t *a, const uint16_t *b, const int32_t *parent,
                            const int32_t *slot, const int32_t *accepted, float *state,
                            float *conv_cache, float *o, int32_t *d_status, cudaStream_t stream);

/* Bytes of workspace lbx_accept_walk needs (0 on bad sizes).  It must be
 * zero-filled once before its first use (it holds one arrival counter per
 * request, which every call that runs to completion leaves at zero, and the
 * per-slice partial results); two calls that run at the same time must not
 * share it. */
size_t lbx_accept_workspace_size(int Bq, int N, int V);

/*
 * Verify argmax and greedy acceptance walk, on the device (Lucebox hub README,
 * "GPU draft top-K & verify-argmax (DFlash)": the target's per-node argmax is
 * taken from the logits buffer in place, so no vocabulary x nodes copy goes to
 * the host; greedy decoding, per the same README's serving notes, is the
 * high-acceptance mode).  Its accepted[] output feeds lbx_verify_step /
 * lbx_tree_persist directly, with no host round trip.
 *   logits [Bq][N][V] fp32 (4-byte aligned): the target's scores after each
 *     node (row n = the distribution of the token that follows node n);
 *   draft [Bq][N] int32: the draft token each node carries (node 0, the
 *     root = the last accepted token, is not read); parent [Bq][N] int32 as
 *     for lbx_verify_step (parent[0] = -1, parent[i] in [0, i));
 *   argmax_out [Bq][N] int32 (may be NULL): the target's choice at each node,
 *     the index of the largest logit, NaN ranking below every number, the
 *     lowest index among equal values (and in an all-NaN row);
 *   accepted_out [Bq] int32: the node where the walk stops -- from the root,
 *     repeatedly step to the lowest-index child whose draft token equals the
 *     target's choice at the current node;
 *   next_out [Bq] int32: the target's choice at the accepted node (the token
 *     that follows the accepted path).
 * All pointers are device pointers owned by the caller; the call is
 * asynchronous on `stream`.  Returns LBX_EINVAL for bad sizes (N >
 * LBX_ACCEPT_MAX_NODES), NULL or misaligned pointers or a short workspace,
 * LBX_ECUDA if the launch fails.  A request whose parent array breaks the
 * tree rules stores LBX_ETREE in *d_status (if not NULL) and writes none of
 * its outputs.  Draft tokens outside [0, V) never match.
 */
int lbx_accept_walk(int Bq, int N, int V, const float *logits, const int32_t *draft,
                    const int32_t *parent, int32_t *argmax_out, int32_t *accepted_out,
                    int32_t *next_out, void *workspace, size_t workspace_bytes,
                    int32_t *d_status, cudaStream_t stream);

/*
 * DDTree construction from the draft's top-K scores, on the device (Lucebox
 * hub README: DDTree, the tree-structured verify that beats chain verify at
 * the same budget, in "Algorithms used"; budget 22 on the RTX 3090 in
 * "Implemented here"; the draft's per-position top-K tokens, K in 1..8, in
 * "GPU draft top-K & verify-argmax (DFlash)").  The output parent array is
 * topologically numbered and feeds lbx_verify_step as is.
 *   logp [Bq][D][K] fp32: log-probabilities of the draft's top-K tokens at
 *     each of the D positions after the root (any order within a position;
 *     -inf allowed, NaN not);
 *   tok [Bq][D][K] int32: those tokens; root_tok [Bq] int32: the root's
 *     token (the last accepted token);
 *   parent_out, token_out [Bq][B] int32; depth_out [Bq][B] int32 and
 *     score_out [Bq][B] fp32 may be NULL; n_nodes_out [Bq] int32.
 * A node's score is the sum of the log-probabilities on its path, added in
 * fp32 from the root down; the tree is built best first: from the root
 * (score 0) the not-yet-added child of an added node with the highest score
 * joins next -- ties: the lower parent index, then the lower k -- until B
 * nodes or no candidate is left (n_nodes < B only when the whole trie of
 * depth D has fewer nodes).  Nodes are numbered in joining order; unused
 * slots get parent, token and depth -1 and score 0.  Device pointers owned
 * by the caller; asynchronous on `stream`.  Returns LBX_EINVAL for sizes
 * outside 1 <= B <= LBX_MAX_TREE_NODES, 1 <= K <= LBX_DDTREE_MAX_K,
 * 0 <= D <= LBX_DDTREE_MAX_DEPTH or NULL / misaligned pointers, LBX_ECUDA
 * if the launch fails.
 */
int lbx_ddtree_build(int Bq, int D, int K, int B, const float *logp, const int32_t *tok,
                     const int32_t *root_tok, int32_t *parent_out, int32_t *token_out,
                     int32_t *depth_out, float *score_out, int32_t *n_nodes_out,
                     cudaStream_t stream);

/* Bytes of workspace lbx_tree_attention needs for these shapes (0 if they
 * are not supported).  It must be zero-filled once before its first use;
 * every call that runs to completion leaves its counters at zero again; two
 * calls that run at the same time must not share a workspace. */
size_t lbx_attn_workspace_size(int L, int Bq, int N, int Hq, int Hkv, int dh, int T);

/*
 * Tree-masked attention of the hybrid target's full-attention layers in the
 * verify forward (Lucebox hub README: DDTree verifies the whole draft tree in
 * one target forward, "Algorithms used"; the full-attention layers keep a KV
 * cache, "--max-ctx N", and attend to all of it by default, "--fa-window N"
 * = 0).  Draft node n sits one position after its parent, so its query sees
 * the request's cached context and the tree nodes on its own root path
 * (its ancestors and itself):
 *     o[l][b][n][hq] = sum_j softmax_j(scale * q[l][b][n][hq] . k_j) v_j,
 * over j in { cache positions 0 .. ctx_len[b]-1 } u { tree nodes on the path
 * root -> n }, with KV head g = hq / (Hq/Hkv) (contiguous GQA groups).
 * Layers are a batch dimension sharing the tree and the context lengths.
 *   q        [L][Bq][N][Hq][dh]   bf16
 *   k_cache, v_cache [L][Bq][T][Hkv][dh] bf16 (T = capacity; may be NULL
 *            when T == 0); positions at or past ctx_len[b] are never used
 *   k_tree, v_tree   [L][Bq][N][Hkv][dh] bf16: the tree nodes' own keys and
 *            values (already projected and position-encoded by the caller)
 *   ctx_len  [Bq] int32 in 0..T;  parent [Bq][N] int32 (the draft tree)
 *   o        [L][Bq][N][Hq][dh]   fp32 out
 *   scale    > 0, finite (1/sqrt(dh) for plain scaled dot-product attention)
 * dh must be LBX_ATTN_HEAD_DIM and 1 <= N <= LBX_ATTN_MAX_NODES; Hq % Hkv ==
 * 0.  Computed on the tensor cores: S = Q K^T per key block and O += P V with
 * bf16 operands (P split into hi + lo) and fp32 accumulation, softmax in
 * fp32.  Device pointers owned by the caller (bf16 arrays and o 16-byte
 * aligned); asynchronous on `stream`.  Returns LBX_EINVAL for unsupported
 * shapes, NULL or misaligned pointers or a short workspace, LBX_ECUDA if the
 * launch fails; an invalid tree or a ctx_len outside 0..T is reported as
 * LBX_ETREE through d_status (nullable) and nothing is written.
 */
int lbx_tree_attention(int L, int Bq, int N, int Hq, int Hkv, int dh, int T, float scale,
                       const int32_t *ctx_len, const int32_t *parent, const uint16_t *q,
                       const uint16_t *k_cache, const uint16_t *v_cache, const uint16_t *k_tree,
                       const uint16_t *v_tree, float *o, void *workspace, size_t workspace_bytes,
                       int32_t *d_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LBX_H */
