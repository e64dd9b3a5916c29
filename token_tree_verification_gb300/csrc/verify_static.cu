// spec_tree_verify_static: tree verification for callers that cannot
// allocate device memory.
//
// Some hosts hand this library only the buffers of a step: a plugin slot in
// an inference engine that owns every byte of device memory and offers no
// allocation hook, or a binding from a runtime that has no CUDA allocator of
// its own.  For them the verification scratch (arrival counters, per-node
// acceptance flags and fallback tokens) lives in one fixed array inside the
// library instead of a caller-provided workspace.  The array is a module
// global, so every GPU that loads the library holds it until the process
// exits; its size bounds the batch this entry point accepts.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/spec_tree.h"

// The scratch itself.  Host code sees only a stand-in symbol: the device
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char spec_verify_scratch[SPEC_VERIFY_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void *g_scratch[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up on the
// first call made with that device current.
int scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_setup_lock);
  if (g_scratch[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, spec_verify_scratch) != cudaSuccess || p == nullptr)
      return SPEC_ERR_CUDA;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_tree_verify_static(const float *target_logits, const float *draft_logits,
                                       const int32_t *tokens, const int32_t *parents,
                                       const int32_t *tree_offsets, int B, int T, int V,
                                       float temperature, uint64_t seed, int32_t *accept_len,
                                       int32_t *path_nodes, int32_t *out_tokens,
                                       int32_t *near_ties, int max_depth_plus1, int32_t *status,
                                       void *stream) {
  // The size limit is checked before anything touches the device.
  const size_t need = spec_tree_verify_workspace_size(B, T, V);
  if (need > SPEC_VERIFY_STATIC_SCRATCH_BYTES) return SPEC_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != SPEC_OK) return rc;
  // The previous call's contents stay in the array; the counters must start
  // at zero, so the part this call uses is cleared on its stream first.
  if (need > 0 &&
      cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return spec_tree_verify(target_logits, draft_logits, tokens, parents, tree_offsets, B, T, V,
                          temperature, seed, accept_len, path_nodes, out_tokens, near_ties,
                          max_depth_plus1, scratch, SPEC_VERIFY_STATIC_SCRATCH_BYTES, status,
                          stream);
}
