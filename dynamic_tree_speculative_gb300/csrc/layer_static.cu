// spec_tree_layer_static: the layer-by-layer builder with its per-tree state in
// a fixed device array inside this library, for callers that cannot allocate
// device memory (include/spec_tree.h says who and why).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_tree.h"
#include "st_kernels.h"

namespace {

constexpr int MAX_DEVICES = 64;
// bytes reserved per tree; the builder's state (about 51 KB) must fit
constexpr size_t SLOT_BYTES = 56 * 1024;

// Every GPU that loads the library holds this array until the process exits.
// Host code sees only a host-side stand-in under this name; kernels get the
// device address looked up by scratch_address().
static __device__ __align__(256) unsigned char layer_scratch[SPEC_TREE_STATIC_MAX_TREES * SLOT_BYTES];

// Device address of layer_scratch on the current device, looked up once per
// device (with that device current) and cached; nullptr if the lookup fails.
void* scratch_address() {
  static void* cache[MAX_DEVICES] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, layer_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    cache[dev] = ptr;
  }
  return cache[dev];
}

}  // namespace

extern "C" int spec_tree_layer_static(const spec_tree_params* p, int B, int V, int layer, int dtype,
                                      const void* layer_logits, int64_t row_stride, const float* u_probe,
                                      const spec_tree_t* tree, int32_t* frontier_token, int32_t* frontier_parent,
                                      uint32_t* status, spec_tree_stream_t stream) {
  if (p == nullptr || B < 0 || B > SPEC_TREE_STATIC_MAX_TREES) return SPEC_TREE_E_PARAM;
  if (st::layer_state_bytes() > SLOT_BYTES) return SPEC_TREE_E_PARAM;  // a build with a larger state
  const bool last = layer == p->depth - 1;
  // the last call also writes the node arrays: check its arguments before
  // anything is launched (B = 0 runs the finish call's checks alone)
  void* const any = reinterpret_cast<void*>(static_cast<uintptr_t>(256));
  if (last) {
    const int rc = spec_tree_finish(p, 0, V, tree, any, status, stream);
    if (rc != SPEC_TREE_OK) return rc;
  }
  if (B == 0) return spec_tree_layer(p, 0, V, layer, dtype, layer_logits, row_stride, u_probe, tree, any,
                                     frontier_token, frontier_parent, status, stream);
  void* const state = scratch_address();
  if (state == nullptr) return SPEC_TREE_E_CUDA;
  int rc = spec_tree_layer(p, B, V, layer, dtype, layer_logits, row_stride, u_probe, tree, state, frontier_token,
                           frontier_parent, status, stream);
  if (rc != SPEC_TREE_OK || !last) return rc;
  return spec_tree_finish(p, B, V, tree, state, status, stream);
}
