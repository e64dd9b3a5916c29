// Step A1: ancestor-or-self bitmask and depth of every tree node.
//
// SpecInfer news write-up, "Token 樹驗證器": the verifier decodes every path of
// the token tree at once through a mask matrix; SpecInfer developer article
// §2.1: each node keeps a parent pointer and the tree_attention mask hides a
// key where the mask is 0.  Here a node's mask row is the set of tree slots it
// may attend to: itself and its ancestors.
//
// One CTA of 128 threads per request; the parent array is staged in shared
// memory, validated, and every thread builds its node's 128-bit set by
// OR-ing in the parent's set level by level (depth <= 127), so each node costs
// O(depth) shared-memory steps and one 16-byte store.
#include "common.cuh"

namespace spec {

__global__ void __launch_bounds__(SPEC_MAX_TREE_NODES)
build_tree_mask_kernel(const int32_t *__restrict__ parents, const int32_t *__restrict__ offsets,
                       int B, int T, uint4 *__restrict__ mask, int32_t *__restrict__ depth,
                       int32_t *__restrict__ status) {
  __shared__ int32_t par[SPEC_MAX_TREE_NODES];
  __shared__ uint4 anc[SPEC_MAX_TREE_NODES];
  __shared__ int32_t dep[SPEC_MAX_TREE_NODES];
  __shared__ int bad;
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  const int lo = __ldg(offsets + b), hi = __ldg(offsets + b + 1);
  const int n = hi - lo;
  if (lo < 0 || hi > T || n < 1 || n > SPEC_MAX_TREE_NODES) {
    if (i == 0) report(status, b, SPEC_ERR_TREE_TOO_LARGE);
    return;
  }
  if (i == 0) bad = 0;
  __syncthreads();
  if (i < n) {
    const int p = in_bounds(lo + i, T, status, b) ? __ldg(parents + lo + i) : -2;
    par[i] = p;
    const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
    if (!ok) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (i == 0) report(status, b, SPEC_ERR_BAD_PARENT);
    return;
  }
  // Level-synchronous propagation: after round r every node of depth <= r
  // holds its final set.  A node is final once its parent is final.
  uint4 m = make_uint4(0, 0, 0, 0);
  if (i < n) {
    (&m.x)[i >> 5] = 1u << (i & 31);
    anc[i] = m;
    dep[i] = (i == 0) ? 0 : -1;
  }
  __syncthreads();
  for (int round = 0; round < n; ++round) {
    bool changed = false;
    uint4 nm = m;
    int nd = -1;
    if (i < n && i > 0 && dep[i] < 0) {
      const int p = par[i];
      const int dp = dep[p];
      if (dp >= 0) {
        const uint4 pm = anc[p];
        nm.x |= pm.x; nm.y |= pm.y; nm.z |= pm.z; nm.w |= pm.w;
        nd = dp + 1;
        changed = true;
      }
    }
    const int any = __syncthreads_or(changed);
    if (changed) {
      anc[i] = nm;
      dep[i] = nd;
      m = nm;
    }
    __syncthreads();
    if (!any) break;
  }
  if (i < n && in_bounds(lo + i, T, status, b)) {
    mask[lo + i] = anc[i];
    depth[lo + i] = dep[i];
  }
}

}  // namespace spec

extern "C" int spec_build_tree_mask(const int32_t *parents, const int32_t *tree_offsets, int B,
                                    int T, uint32_t *mask, int32_t *depth, int32_t *status,
                                    void *stream) {
  if (!parents || !tree_offsets || !mask || !depth || !status) return SPEC_ERR_NULL;
  if (B < 1 || T < 1 || T > B * SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(mask) & 15) return SPEC_ERR_ALIGNMENT;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(SPEC_MAX_TREE_NODES, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  spec::pdl_attribute(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, spec::build_tree_mask_kernel, parents, tree_offsets, B, T, reinterpret_cast<uint4 *>(mask), depth, status) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}
