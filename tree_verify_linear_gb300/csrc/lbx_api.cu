// lbx_api.cu -- the C ABI: host-side argument checks and kernel dispatch.
#include <math.h>
#include <stdint.h>

#include "gdn_launch.h"
#include "gdn_step.cuh"
#include "lbx.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Shape checks shared by every entry point.
int check_cfg(const lbx_cfg *c) {
  if (!c) return LBX_EINVAL;
  if (c->L < 1 || c->Bq < 1 || c->N < 1 || c->Hk < 1 || c->Hv < 1) return LBX_EINVAL;
  if (c->Hv % c->Hk != 0) return LBX_EINVAL;
  if (c->d != 32 && c->d != 64 && c->d != 128) return LBX_EINVAL;
  if (c->K < 1 || c->K > LBX_MAX_CONV_WIDTH) return LBX_EINVAL;
  if (c->n_slots < c->Bq) return LBX_EINVAL;
  if (!(c->l2_eps >= 0.0f) || !isfinite(c->l2_eps) || !isfinite(c->q_scale)) return LBX_EINVAL;
  // 32-bit index headroom used by the kernels
  if ((long long)c->Bq * c->N > (1LL << 30)) return LBX_EINVAL;
  if ((long long)(2 * c->Hk + c->Hv) * c->d > (1LL << 24)) return LBX_EINVAL;
  if ((long long)c->L * c->Bq * c->Hv * 4 > 0x7fffffffLL) return LBX_EINVAL;
  return LBX_OK;
}

bool ok16(const void *p) { return p != nullptr && aligned(p, 16); }
bool ok4(const void *p) { return p != nullptr && aligned(p, 4); }
bool ok2(const void *p) { return p != nullptr && aligned(p, 2); }
// With conv width 1 there is no conv cache; its pointer may then be NULL.
bool cache_ok(const lbx_cfg *c, const void *p, uintptr_t a) {
  return (c->K == 1 && p == nullptr) || (p != nullptr && aligned(p, a));
}

// The mode a verify step runs in (LBX_MODE_AUTO resolved).
int resolve_mode(const lbx_cfg *c) {
  if (c->mode == LBX_MODE_AUTO) return c->N <= LBX_MAX_TREE_NODES ? LBX_MODE_TREE : LBX_MODE_CHUNKED;
  return c->mode;
}

// Whether lbx_verify_step runs the tensor-core step for this configuration.
bool uses_tc(const lbx_cfg *c) {
  return resolve_mode(c) == LBX_MODE_TREE && lbx::step_tc_supported(c->d, c->N, 0);
}

lbx::StepArgs step_args(const lbx_cfg *c) {
  lbx::StepArgs A = {};
  A.L = c->L, A.Bq = c->Bq, A.N = c->N, A.Hk = c->Hk, A.Hv = c->Hv, A.K = c->K;
  A.n_slots = c->n_slots;
  A.l2_eps = c->l2_eps;
  A.q_scale = c->q_scale;
  return A;
}

}  // namespace

namespace lbx {
size_t counters_bytes(int L, int Bq, int Hk) {
  const size_t counters = (size_t)L * Bq * Hk * sizeof(unsigned int);
  return (counters + 255) & ~(size_t)255;
}
}  // namespace lbx

extern "C" {

const char *lbx_strerror(int status) {
  switch (status) {
    case LBX_OK: return "ok";
    case LBX_EINVAL: return "invalid argument (dimension, pointer, alignment, limit or index)";
    case LBX_ECUDA: return "CUDA launch or runtime error";
    case LBX_ETREE: return "invalid draft tree (parent array is not a topologically numbered tree, or not a chain in chunked mode)";
    case LBX_ETIMEOUT: return "a bounded wait inside a kernel gave up (reported through d_status)";
  }
  return "unknown status";
}

size_t lbx_workspace_size(const lbx_cfg *cfg) {
  if (check_cfg(cfg) != LBX_OK) return 0;
  size_t n = lbx::counters_bytes(cfg->L, cfg->Bq, cfg->Hk);
  if (uses_tc(cfg)) {
    const size_t tc = lbx::step_tc_workspace_bytes(cfg->L, cfg->Bq, cfg->Hk, cfg->Hv, cfg->N);
    n = tc > n ? tc : n;
  }
  return n;
}

int lbx_tree_conv(const lbx_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                  const float *conv_cache, const int32_t *parent, const int32_t *slot,
                  float *qkv_out, int32_t *d_status, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (cfg->N > LBX_MAX_TREE_NODES) return LBX_EINVAL;
  if (!ok16(x) || !ok16(conv_w) || !cache_ok(cfg, conv_cache, 16) || !ok4(parent) ||
      !ok4(slot) || !ok16(qkv_out) || (d_status && !aligned(d_status, 4)))
    return LBX_EINVAL;
  lbx::ConvArgs A = {};
  A.L = cfg->L, A.Bq = cfg->Bq, A.N = cfg->N, A.Hk = cfg->Hk, A.Hv = cfg->Hv, A.K = cfg->K;
  A.n_slots = cfg->n_slots;
  A.l2_eps = cfg->l2_eps;
  A.x = x, A.conv_w = conv_w, A.conv_cache = conv_cache, A.parent = parent, A.slot = slot;
  A.qkv = qkv_out, A.status = d_status;
  return lbx::launch_tree_conv(A, cfg->d, stream);
}

int lbx_tree_deltanet(const lbx_cfg *cfg, const float *qkv, const uint16_t *a, const uint16_t *b,
                      const float *state, const int32_t *parent, const int32_t *slot, float *o,
                      float *node_states, int32_t *d_status, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (cfg->N > LBX_MAX_TREE_NODES) return LBX_EINVAL;
  if (!ok16(qkv) || !ok2(a) || !ok2(b) || !ok16(state) || !ok4(parent) || !ok4(slot) ||
      !ok16(o) || (node_states && !aligned(node_states, 16)) ||
      (d_status && !aligned(d_status, 4)))
    return LBX_EINVAL;
  lbx::StepArgs A = step_args(cfg);
  A.chain = 0;
  A.cap = cfg->N;
  A.qkv = qkv, A.a = a, A.b = b, A.state_in = state, A.parent = parent, A.slot = slot;
  A.o = o, A.node_states = node_states, A.status = d_status;
  return lbx::launch_step_unfused(A, cfg->d, stream);
}

int lbx_tree_persist(const lbx_cfg *cfg, const uint16_t *x, const float *node_states,
                     const int32_t *parent, const int32_t *slot, const int32_t *accepted,
                     float *state, float *conv_cache, int32_t *d_status, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (cfg->N > LBX_MAX_TREE_NODES) return LBX_EINVAL;
  if (!ok2(x) || !ok16(node_states) || !ok4(parent) || !ok4(slot) || !ok4(accepted) ||
      !ok16(state) || !cache_ok(cfg, conv_cache, 4) || (d_status && !aligned(d_status, 4)))
    return LBX_EINVAL;
  lbx::PersistArgs A = {};
  A.L = cfg->L, A.Bq = cfg->Bq, A.N = cfg->N, A.Hk = cfg->Hk, A.Hv = cfg->Hv, A.K = cfg->K;
  A.n_slots = cfg->n_slots;
  A.x = x, A.node_states = node_states, A.parent = parent, A.slot = slot, A.accepted = accepted;
  A.state = state, A.conv_cache = conv_cache, A.status = d_status;
  return lbx::launch_tree_persist(A, cfg->d, stream);
}

int lbx_verify_step(const lbx_cfg *cfg, const uint16_t *x, const uint16_t *conv_w,
                    const uint16_t *a, const uint16_t *b, const int32_t *parent,
                    const int32_t *slot, const int32_t *accepted, float *state, float *conv_cache,
                    float *o, void *workspace, size_t workspace_bytes, int32_t *d_status,
                    cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  const int mode = resolve_mode(cfg);
  if (mode != LBX_MODE_TREE && mode != LBX_MODE_CHUNKED && mode != LBX_MODE_TREE_CUDA_CORES)
    return LBX_EINVAL;
  if (mode != LBX_MODE_CHUNKED && cfg->N > LBX_MAX_TREE_NODES) return LBX_EINVAL;
  if (!ok16(x) || !ok16(conv_w) || !ok2(a) || !ok2(b) || !ok4(parent) || !ok4(slot) ||
      !ok4(accepted) || !ok16(state) || !cache_ok(cfg, conv_cache, 16) || !ok16(o) || !ok4(workspace) ||
      (d_status && !aligned(d_status, 4)))
    return LBX_EINVAL;
  if (workspace_bytes < lbx_workspace_size(cfg)) return LBX_EINVAL;
  lbx::StepArgs A = step_args(cfg);
  A.chain = mode == LBX_MODE_CHUNKED;
  A.cap = A.chain ? (cfg->N < LBX_CHAIN_CHUNK ? cfg->N : LBX_CHAIN_CHUNK) : cfg->N;
  A.x = x, A.conv_w = conv_w, A.conv_cache = conv_cache, A.a = a, A.b = b;
  A.parent = parent, A.slot = slot, A.accepted = accepted;
  A.state_in = state, A.state_out = state, A.conv_cache_out = conv_cache;
  A.o = o, A.counters = static_cast<unsigned int *>(workspace), A.status = d_status;
  if (uses_tc(cfg)) return lbx::launch_step_tc(A, workspace, workspace_bytes, stream);
  if (A.chain && lbx::chain_tc_supported(cfg->d)) return lbx::launch_chain_tc(A, stream);
  return lbx::launch_step_fused(A, cfg->d, stream);
}

}  // extern "C"
