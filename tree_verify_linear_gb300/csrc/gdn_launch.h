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

// Tensor-core fused step (d = 128, tree mode, N <= 24).
bool step_tc_supported(int d, int N, int chain);
int launch_step_tc(const StepArgs &A, cudaStream_t st);

// Row-block size and product-tile width used for head dimension d and node
// capacity cap; returns the dynamic shared memory bytes (0 if unsupported).
int step_smem_bytes(int d, int cap);

}  // namespace lbx
