// Steps V1-V4 and R for greedy verification, one CTA per node.
//
// Sources: speculative-decoding explainer (intelliparadigm.com) §2.2
// 三阶段工作流程详解 (stage 1 drafts greedily); SpecInfer developer article
// §2.1 (accept the longest verified prefix).
//
// The CTA's threads stream the node's target row (the first batch of loads
// is issued before the tree is read) and reduce its argmax, lowest index on
// ties; the node's children are accepted iff their token equals it, and the
// last CTA of a request walks it.  Up to one node per SM: 1024 threads, one
// CTA per SM; more nodes: 256 threads, four CTAs per SM, so one CTA's fixed
// costs (tree, reduction, arrival) overlap the others' row loads.
#include "verify_common.cuh"

namespace spec {

// ---------------------------------------------------------------- greedy
constexpr int kGreedyPrefetch = 8;  // float4 loads per thread issued before the tree is read

template <int kGreedyThreads>
__global__ void __launch_bounds__(kGreedyThreads, 1024 / kGreedyThreads)
tree_verify_greedy_node_kernel(const VerifyArgs a) {
  constexpr int kGW = kGreedyThreads / 32;
  __shared__ TreeSmem ts;
  __shared__ float rv[kGW];
  __shared__ int ri[kGW];
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const float *row = a.target + static_cast<size_t>(t) * a.V;
  const bool vec = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0);
  const int n4 = vec ? a.V >> 2 : 0;
  pdl_trigger();
  pdl_wait();
  const TreeLoads tl = tree_loads(a, t);
  // first batch of the row, in flight while the tree is read
  float4 pre[kGreedyPrefetch];
#pragma unroll
  for (int e = 0; e < kGreedyPrefetch; ++e) {
    const int i = tid + e * kGreedyThreads;
    pre[e] = i < n4 ? __ldcs(reinterpret_cast<const float4 *>(row) + i)
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  const NodeCtx c = load_tree(a, t, ts, tl);
  if (!c.err) {
    ArgMax am{-INFINITY, 0x7fffffff};
    if (vec) {
#pragma unroll
      for (int e = 0; e < kGreedyPrefetch; ++e) {
        const int i = tid + e * kGreedyThreads;
        if (i < n4) {
          am = better(am, ArgMax{pre[e].x, 4 * i});
          am = better(am, ArgMax{pre[e].y, 4 * i + 1});
          am = better(am, ArgMax{pre[e].z, 4 * i + 2});
          am = better(am, ArgMax{pre[e].w, 4 * i + 3});
        }
      }
      for (int i = tid + kGreedyPrefetch * kGreedyThreads; i < n4; i += kGreedyThreads) {
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(row) + i);
        am = better(am, ArgMax{v.x, 4 * i});
        am = better(am, ArgMax{v.y, 4 * i + 1});
        am = better(am, ArgMax{v.z, 4 * i + 2});
        am = better(am, ArgMax{v.w, 4 * i + 3});
      }
    } else {
      for (int i = tid; i < a.V; i += kGreedyThreads) am = better(am, ArgMax{__ldcs(row + i), i});
    }
    am = warp_argmax(am);
    if (lane == 0) {
      rv[w] = am.v;
      ri[w] = am.i;
    }
    __syncthreads();
    if (tid == 0) {
      ArgMax g{rv[0], ri[0]};
      for (int i = 1; i < kGW; ++i) g = better(g, ArgMax{rv[i], ri[i]});
      a.fallback[t] = g.i;
      bool accepted = false;
      for (int j = 0; j < c.k; ++j) {
        const int ch = ts.child[j];
        const bool hit = ts.tok[ch] == g.i;
        if (in_bounds(c.lo + ch, a.T, a.status, c.b)) a.flags[c.lo + ch] = hit ? kFlagAccept : 0;
        accepted |= hit;
      }
      ts.stop_fb = accepted ? -1 : g.i;   // -1: the walk goes on below this node
    }
  } else if (tid == 0 && c.b >= 0) {
    report(a.status, c.b, c.err);
  }
  __syncthreads();  // the node's flags and fallback are written
  arrive_and_walk(a, c, ts, c.err ? -1 : ts.stop_fb, 0, false);
}

int launch_verify_greedy(const VerifyArgs &args, cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool wide = args.T <= sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(args.T), 1, 1);
  cfg.blockDim = dim3(wide ? 1024 : 256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  pdl_attribute(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = wide ? cudaLaunchKernelEx(&cfg, tree_verify_greedy_node_kernel<1024>, args)
                             : cudaLaunchKernelEx(&cfg, tree_verify_greedy_node_kernel<256>, args);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace spec
