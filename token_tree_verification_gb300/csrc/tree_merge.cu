// Merging two speculators' token trees into one (SpecInfer developer
// article, §7.2 混合推测策略: an LLM speculator's tree merged with an n-gram
// speculator's, tree.merge(other)), on the device: one CTA per request.
//
// A's nodes keep their indices; each node of B whose token path from the
// shared root is already present maps to the present node of lowest merged
// index, and the others are appended in B's order.  The CTA resolves B level
// by level: a node's representative is the A node with the same parent
// representative and token (lowest index), else the first B node of its
// level with the same parent representative and token (n_a + its index).
// Representatives never depend on merged indices, so the level loop needs no
// prefix sums; one scan over B's new nodes then gives their merged indices.
#include "common.cuh"

namespace spec {

namespace {
constexpr int kMergeThreads = 256;
constexpr int kMergeCap = SPEC_MAX_TREE_NODES;

struct MergeSmem {
  int pa[kMergeCap], ta[kMergeCap], pb[kMergeCap], tb[kMergeCap];
  int db[kMergeCap];       // depth of B's nodes
  int rep[kMergeCap];      // B node -> representative (A index, or n_a + first B index)
  int idx[kMergeCap];      // B node -> merged index
  int scan[kMergeCap];
  int err, maxd;
};
}  // namespace

__global__ void __launch_bounds__(kMergeThreads)
tree_merge_kernel(const int32_t *parents_a, const int32_t *tokens_a, const int32_t *off_a,
                  const int32_t *parents_b, const int32_t *tokens_b, const int32_t *off_b, int B,
                  int Ta, int Tb, int32_t *out_parents, int32_t *out_tokens, int32_t *map_b,
                  int32_t *n_out, int32_t *status) {
  __shared__ MergeSmem sm;
  const int b = blockIdx.x, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  const int lo_a = __ldg(off_a + b), hi_a = __ldg(off_a + b + 1);
  const int lo_b = __ldg(off_b + b), hi_b = __ldg(off_b + b + 1);
  const int na = hi_a - lo_a, nb = hi_b - lo_b;
  if (na < 1 || na > kMergeCap || nb < 1 || nb > kMergeCap || lo_a < 0 || hi_a > Ta || lo_b < 0 ||
      hi_b > Tb) {
    if (tid == 0) report(status, b, SPEC_ERR_TREE_TOO_LARGE);
    return;
  }
  if (tid == 0) {
    sm.err = 0;
    sm.maxd = 0;
  }
  for (int i = tid; i < kMergeCap; i += kMergeThreads) {
    if (i < na) {
      const bool in = in_bounds(lo_a + i, Ta, status, b);
      sm.pa[i] = in ? __ldg(parents_a + lo_a + i) : -2;
      sm.ta[i] = in ? __ldg(tokens_a + lo_a + i) : -1;
    }
    if (i < nb) {
      const bool in = in_bounds(lo_b + i, Tb, status, b);
      sm.pb[i] = in ? __ldg(parents_b + lo_b + i) : -2;
      sm.tb[i] = in ? __ldg(tokens_b + lo_b + i) : -1;
    }
  }
  __syncthreads();
  // parents: -1 at the root, in [0, i) elsewhere, in both trees
  for (int i = tid; i < kMergeCap; i += kMergeThreads) {
    bool bad = false;
    if (i < na) bad |= i == 0 ? sm.pa[0] != -1 : (sm.pa[i] < 0 || sm.pa[i] >= i);
    if (i < nb) bad |= i == 0 ? sm.pb[0] != -1 : (sm.pb[i] < 0 || sm.pb[i] >= i);
    if (bad) atomicExch(&sm.err, SPEC_ERR_BAD_PARENT);
  }
  __syncthreads();
  if (sm.err) {
    if (tid == 0) report(status, b, sm.err);
    return;
  }
  // depths of B's nodes (parents are valid: each walk ends at the root)
  for (int i = tid; i < nb; i += kMergeThreads) {
    int d = 0;
    for (int x = i; x > 0; x = sm.pb[x]) ++d;
    sm.db[i] = d;
    atomicMax(&sm.maxd, d);
    sm.rep[i] = 0;   // the roots coincide
  }
  __syncthreads();
  const int maxd = sm.maxd;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kMergeThreads / 32;
  for (int d = 1; d <= maxd; ++d) {
    // one warp per node of this level; its lanes search A's nodes, then B's
    // earlier nodes, four at a time (the lowest index wins)
    for (int i = warp; i < nb; i += kWarps) {
      if (sm.db[i] != d) continue;
      const int pr = sm.rep[sm.pb[i]];   // resolved at level d - 1
      const int tk = sm.tb[i];
      int r = -1;
#pragma unroll
      for (int s = 0; s < kMergeCap / 32 && r < 0; ++s) {
        const int j = s * 32 + lane;
        const bool hit = pr < na && j >= 1 && j < na && sm.pa[j] == pr && sm.ta[j] == tk;
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (m) r = s * 32 + __ffs(m) - 1;
      }
#pragma unroll
      for (int s = 0; s < kMergeCap / 32 && r < 0; ++s) {
        // the first node of this level of B with the same parent and token
        const int i2 = s * 32 + lane;
        const bool hit = i2 >= 1 && i2 <= i && sm.db[i2] == d && sm.tb[i2] == tk &&
                         sm.rep[sm.pb[i2]] == pr;
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (m) r = na + s * 32 + __ffs(m) - 1;
      }
      if (lane == 0) sm.rep[i] = r;
    }
    __syncthreads();
  }
  // merged indices: A's nodes, then B's new nodes in B's order
  for (int i = tid; i < nb; i += kMergeThreads) sm.scan[i] = (i > 0 && sm.rep[i] == na + i) ? 1 : 0;
  __syncthreads();
  if (tid < 32) {
    // exclusive scan over at most 128 flags, four per lane
    int v[4], tot = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = tid * 4 + s;
      v[s] = i < nb ? sm.scan[i] : 0;
      tot += v[s];
    }
    int inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (tid >= o) inc += y;
    }
    int run = inc - tot;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = tid * 4 + s;
      if (i < nb) sm.idx[i] = na + run;
      run += v[s];
    }
    if (tid == 31) sm.maxd = na + inc;   // the merged node count
  }
  __syncthreads();
  const int n = sm.maxd;
  if (n > kMergeCap) {
    if (tid == 0) report(status, b, SPEC_ERR_TREE_TOO_LARGE);
    return;
  }
  // each B node's merged index: its representative's
  for (int i = tid; i < nb; i += kMergeThreads) {
    const int r = sm.rep[i];
    sm.scan[i] = r < na ? r : sm.idx[r - na];
  }
  __syncthreads();
  int32_t *op = out_parents + static_cast<size_t>(b) * kMergeCap;
  int32_t *ot = out_tokens + static_cast<size_t>(b) * kMergeCap;
  int32_t *mb = map_b + static_cast<size_t>(b) * kMergeCap;
  for (int j = tid; j < kMergeCap; j += kMergeThreads) {
    if (j >= n) {
      op[j] = -2;
      ot[j] = -1;
    } else if (j < na) {
      op[j] = sm.pa[j];
      ot[j] = sm.ta[j];
    }
    mb[j] = j < nb ? sm.scan[j] : -1;
  }
  for (int i = tid; i < nb; i += kMergeThreads) {
    if (i > 0 && sm.rep[i] == na + i) {
      const int j = sm.idx[i];
      if (in_bounds(j, kMergeCap, status, b)) {
        op[j] = sm.scan[sm.pb[i]];
        ot[j] = sm.tb[i];
      }
    }
  }
  if (tid == 0) n_out[b] = n;
}

}  // namespace spec

extern "C" int spec_tree_merge(const int32_t *parents_a, const int32_t *tokens_a,
                               const int32_t *offsets_a, const int32_t *parents_b,
                               const int32_t *tokens_b, const int32_t *offsets_b, int B, int Ta,
                               int Tb, int32_t *out_parents, int32_t *out_tokens, int32_t *map_b,
                               int32_t *n_out, int32_t *status, void *stream) {
  if (!parents_a || !tokens_a || !offsets_a || !parents_b || !tokens_b || !offsets_b ||
      !out_parents || !out_tokens || !map_b || !n_out || !status)
    return SPEC_ERR_NULL;
  if (B < 1 || Ta < B || Tb < B || Ta > B * SPEC_MAX_TREE_NODES || Tb > B * SPEC_MAX_TREE_NODES)
    return SPEC_ERR_SHAPE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(spec::kMergeThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  spec::pdl_attribute(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, spec::tree_merge_kernel, parents_a, tokens_a, offsets_a,
                            parents_b, tokens_b, offsets_b, B, Ta, Tb, out_parents, out_tokens,
                            map_b, n_out, status) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}
