// gdn_launch.h -- host-side launchers of the tree-verify kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lbx.h"

namespace lbx {

struct StepArgs;

struct ConvArgs {
  int L, Bq, N, Hk, Hv, K, n_slots;
  float l2_eps;
  const uint16_t *x, *conv_w;
  const float *conv_cache;
  const int32_t *parent, *slot;
  float *qkv;
  int32_t *status;
};

struct PersistArgs {
  int L, Bq, N, Hk, Hv, K, n_slots;
  const uint16_t *x;
  const float *node_states;
  const int32_t *parent, *slot, *accepted;
  float *state, *conv_cache;
  int32_t *status;
};

int launch_tree_conv(const ConvArgs &A, int d, cudaStream_t st);
int launch_tree_persist(const PersistArgs &A, int d, cudaStream_t st);

// Fused conv + recurrence + persist (tree or chunked chain).
int launch_step_fused(const StepArgs &A, int d, cudaStream_t st);
// Recurrence from a conv output; node_states written when A.node_states != NULL.
int launch_step_unfused(const StepArgs &A, int d, cudaStream_t st);

// Tensor-core fused step (d = 128, tree mode, N <= 24): a prep kernel per key
// head, then the step kernel.  Its workspace holds the prep kernel's tables
// and records (step_tc_workspace_bytes); no arrival counters.
bool step_tc_supported(int d, int N, int chain);
size_t step_tc_workspace_bytes(int L, int Bq, int Hk, int Hv, int N);
int launch_step_tc(const StepArgs &A, void *ws, size_t ws_bytes, cudaStream_t st);

// Tensor-core chunked step for chains (d = 128): one CTA per (layer,
// request, value head) sequence, 16-token chunks, arrival counters in the
// workspace as for the CUDA-core kernels.
bool chain_tc_supported(int d);
int launch_chain_tc(const StepArgs &A, cudaStream_t st);

// Workspace of the CUDA-core fused step: one arrival counter per (layer,
// request, key head), 256-byte rounded.
size_t counters_bytes(int L, int Bq, int Hk);

// Row-block size and product-tile width used for head dimension d and node
// capacity cap; returns the dynamic shared memory bytes (0 if unsupported).
int step_smem_bytes(int d, int cap);

}  // namespace lbx
