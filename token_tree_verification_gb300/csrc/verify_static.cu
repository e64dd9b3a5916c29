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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "verify_common.cuh"

// The scratch itself.  Host code sees only a stand-in symbol: the device
// address is looked up with cudaGetSymbolAddress, with the device current.
static __device__ __align__(256) unsigned char spec_verify_scratch[SPEC_VERIFY_STATIC_SCRATCH_BYTES];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct ScratchSlot {
  unsigned long long ctx_id;   // the context the address belongs to (0: none yet)
  void *ptr;
};

std::mutex g_setup_lock;
ScratchSlot g_scratch[spec::kMaxDevices] = {};

// Identity of the context current on this thread: the driver's unique
// context id, so that a context destroyed and created again (a device reset)
// is told apart from the one the cached address belongs to.
bool current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch in the current device's context.  The
// lookup runs on the first call made with that device current, and again
// when the device's context has changed since (after a device reset).
int scratch_on_current_device(void **out) {
  const int dev = spec::current_device();
  if (dev < 0) return SPEC_ERR_CUDA;
  // Before the caller's first runtime call on the device no context may be
  // current yet; the symbol lookup itself binds the device's primary context.
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> guard(g_setup_lock);
  ScratchSlot &slot = g_scratch[dev];
  if (!have_id || slot.ptr == nullptr || slot.ctx_id != id) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, spec_verify_scratch) != cudaSuccess || p == nullptr)
      return SPEC_ERR_CUDA;
    if (!have_id && !current_context_id(&id)) return SPEC_ERR_CUDA;
    slot.ptr = p;
    slot.ctx_id = id;
  }
  *out = slot.ptr;
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
  // The previous call's contents stay in the array and the counters must
  // start at zero: after its host-side checks have passed, the entry clears
  // the part this call uses on `stream`, then launches.
  return spec::verify_entry(target_logits, draft_logits, tokens, parents, tree_offsets, B, T, V,
                            temperature, 1.f, seed, accept_len, path_nodes, out_tokens, near_ties,
                            max_depth_plus1, scratch, SPEC_VERIFY_STATIC_SCRATCH_BYTES, status,
                            stream, true);
}
