// lbx_noalloc.cu -- lbx_verify_step_noalloc: the fused verify step for callers
// that cannot allocate device memory.
//
// lbx_verify_step needs a small workspace (one arrival counter per (layer,
// request, key head)).  Some callers cannot provide it: an engine that
// reserves all device memory for its caches up front and forbids any later
// cudaMalloc (which would also synchronise the device mid-decode), or a plugin
// running inside a host framework that owns the only allocator.  For them the
// counters live in the fixed array below, part of the library's own device
// image: every GPU that loads the library holds it until the process exits.
#include <mutex>

#include "lbx.h"

namespace {

// File-scope device array; in host code its name is only a stand-in, so the
// host never passes it to a kernel directly -- it passes the address that
// cudaGetSymbolAddress returns for the current device.
__device__ __align__(256) unsigned int g_noalloc_counters[LBX_NOALLOC_MAX_GROUPS];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
unsigned int *g_counters_dev[kMaxDevices] = {};

// Device address of the counter array on the current device, looked up once
// per device (with that device current).
int counters_on_current_device(unsigned int **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LBX_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_counters_dev[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_counters) != cudaSuccess || p == nullptr)
      return LBX_ECUDA;
    g_counters_dev[dev] = static_cast<unsigned int *>(p);
  }
  *out = g_counters_dev[dev];
  return LBX_OK;
}

}  // namespace

extern "C" int lbx_verify_step_noalloc(const lbx_cfg *cfg, const uint16_t *x,
                                       const uint16_t *conv_w, const uint16_t *a,
                                       const uint16_t *b, const int32_t *parent,
                                       const int32_t *slot, const int32_t *accepted, float *state,
                                       float *conv_cache, float *o, int32_t *d_status,
                                       cudaStream_t stream) {
  if (cfg == nullptr) return LBX_EINVAL;
  lbx_cfg c = *cfg;
  if (lbx_workspace_size(&c) > sizeof(g_noalloc_counters)) {
    // The tensor-core step keeps per-key-head records in its workspace, far
    // more than the fixed array holds: run the CUDA-core tree kernel, which
    // needs only the counters.
    const int mode = c.mode == LBX_MODE_AUTO
                         ? (c.N <= LBX_MAX_TREE_NODES ? LBX_MODE_TREE : LBX_MODE_CHUNKED)
                         : c.mode;
    if (mode == LBX_MODE_TREE) c.mode = LBX_MODE_TREE_CUDA_CORES;
  }
  const size_t need = lbx_workspace_size(&c);
  if (need == 0) return LBX_EINVAL;
  if (need > sizeof(g_noalloc_counters)) return LBX_EINVAL;  // over the fixed capacity
  unsigned int *counters = nullptr;
  const int rc = counters_on_current_device(&counters);
  if (rc != LBX_OK) return rc;
  // The array keeps whatever the previous call left; the counters this call
  // uses must start at zero.
  if (cudaMemsetAsync(counters, 0, need, stream) != cudaSuccess) return LBX_ECUDA;
  return lbx_verify_step(&c, x, conv_w, a, b, parent, slot, accepted, state, conv_cache, o,
                         counters, need, d_status, stream);
}
