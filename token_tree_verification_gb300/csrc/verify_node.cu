// Steps V1-V4 and R with one CTA per node (vocabulary up to 32768 entries
// for stochastic verification, any size for greedy verification).
//
// Sources: speculative-decoding explainer (intelliparadigm.com) §2.2
// 三阶段工作流程详解 (stage 2: alpha = min(1, p/q); stage 3: stop at the first
// rejection, draw a new target prediction); SpecInfer developer article §2.1
// (accept the longest verified prefix).  The residual chain uses the closed
// form derived in verify.cu: r_j = max(0, p - c_j q) / W(c_j).
//
// Greedy: 1024 threads stream the node's target row (the first batch of
// loads is issued before the tree is read) and reduce its argmax.
// Stochastic: the target row lands in shared memory through one bulk copy
// while the tree is read; the draft row (internal nodes only) is held in
// registers, 64 entries per thread of 512.  Every reduction round is one
// __syncthreads; the inverse-CDF draw searches three levels (one segment
// per warp, one sub-segment per warp, then one warp scans).
#include "verify_common.cuh"

namespace spec {

constexpr int kNW = kNodeThreads / 32;
constexpr int kGW = kGreedyThreads / 32;

struct NodeScratch {
  float f[2][kNW];       // double-buffered warp partials
  float pair[kNW][4];
  float lvl[kNW];
  int pick;
  float cb[2];
  int clamp;
};

// Sum over the CTA; every thread returns the same value (warp partials added
// in warp order).
__device__ __forceinline__ float node_block_sum(float x, NodeScratch &sc, int parity) {
  x = warp_sum(x);
  if ((threadIdx.x & 31) == 0) sc.f[parity][threadIdx.x >> 5] = x;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kNW; ++i) s += sc.f[parity][i];
  return s;
}

// ---------------------------------------------------------------- greedy
constexpr int kGreedyPrefetch = 8;  // float4 loads per thread issued before the tree is read

__global__ void __launch_bounds__(kGreedyThreads, 1)
tree_verify_greedy_node_kernel(const VerifyArgs a) {
  __shared__ TreeSmem ts;
  __shared__ float rv[kGW];
  __shared__ int ri[kGW];
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const float *row = a.target + static_cast<size_t>(t) * a.V;
  const bool vec = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0);
  const int n4 = vec ? a.V >> 2 : 0;
  // first batch of the row, in flight while the tree is read
  float4 pre[kGreedyPrefetch];
#pragma unroll
  for (int e = 0; e < kGreedyPrefetch; ++e) {
    const int i = tid + e * kGreedyThreads;
    pre[e] = i < n4 ? __ldcs(reinterpret_cast<const float4 *>(row) + i)
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  const NodeCtx c = load_tree(a, t, ts);
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
      for (int j = 0; j < c.k; ++j) {
        const int ch = ts.child[j];
        a.flags[c.lo + ch] = (ts.tok[ch] == g.i) ? kFlagAccept : 0;
      }
    }
  } else if (tid == 0 && c.b >= 0) {
    report(a.status, c.b, c.err);
  }
  arrive_and_walk(a, c, ts, gridDim.x);
}

// ---------------------------------------------------------------- stochastic
// First index (or, with `clamp`, last index) among `cnt` partial sums whose
// running sum passes `target`; updates `prefix` to the sum before it.
__device__ __forceinline__ int pick_bucket(const float *sums, int cnt, float target, float &prefix,
                                           bool &clamp) {
  float run = prefix;
  if (!clamp) {
    for (int i = 0; i < cnt; ++i) {
      if (run + sums[i] > target) {
        prefix = run;
        return i;
      }
      run += sums[i];
    }
    clamp = true;  // rounding kept the running sum below the target
  }
  int last = 0;
  float before = prefix;
  run = prefix;
  for (int i = 0; i < cnt; ++i) {
    if (sums[i] > 0.f) {
      last = i;
      before = run;
    }
    run += sums[i];
  }
  prefix = before;
  return last;
}

__global__ void __launch_bounds__(kNodeThreads, 1)
tree_verify_stoch_node_kernel(const VerifyArgs a) {
  extern __shared__ __align__(128) float prow[];   // the node's target row, then p, then weights
  __shared__ TreeSmem ts;
  __shared__ NodeScratch sc;
  __shared__ __align__(8) uint64_t bar;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int V = a.V;
  const float *trow_g = a.target + static_cast<size_t>(t) * V;
  const float *drow_g = a.draft + static_cast<size_t>(t) * V;
  const bool bulk = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (bulk) {
      mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(V) * 4u);
      bulk_copy_g2s(prow, trow_g, static_cast<uint32_t>(V) * 4u, &bar);
    }
  }
  const NodeCtx c = load_tree(a, t, ts);
  const int k = c.k;
  const bool need_draft = !c.err && k > 0;
  float q[kNodeElems];
#pragma unroll
  for (int e = 0; e < kNodeElems; ++e) {
    const int v = tid + e * kNodeThreads;
    q[e] = (need_draft && v < V) ? __ldcs(drow_g + v) : -INFINITY;
  }
  load_children(a, c, t, ts);
  bool timed_out = false;
  if (bulk) {
    if (!mbar_wait(&bar, 0)) timed_out = true;
  } else if (!c.err) {
    for (int v = tid; v < V; v += kNodeThreads) prow[v] = __ldcs(trow_g + v);
  }
  if (timed_out && tid == 0) report(a.status, c.b, SPEC_ERR_TIMEOUT);
  __syncthreads();

  if (!c.err) {
    const float T_ = a.temp, iT = a.inv_temp;
    const float l2s = iT * 1.4426950408889634f;   // exp(x / T) = 2^(x * l2s)
    // ---- V1: max and sum of exp((x - max)/T), per thread then per CTA
    float ml = -INFINITY, md = -INFINITY;
#pragma unroll
    for (int e = 0; e < kNodeElems; ++e) {
      const int v = tid + e * kNodeThreads;
      if (v < V) ml = fmaxf(ml, prow[v]);
      md = fmaxf(md, q[e]);
    }
    float sl = 0.f, sd = 0.f;
#pragma unroll
    for (int e = 0; e < kNodeElems; ++e) {
      const int v = tid + e * kNodeThreads;
      if (v < V) {
        const float el = fast_exp2((prow[v] - ml) * l2s);
        prow[v] = el;
        sl += el;
      }
      const float ed = need_draft ? fast_exp2((q[e] - md) * l2s) : 0.f;
      q[e] = ed;
      sd += ed;
    }
    const float wml = warp_max(ml), wmd = warp_max(md);
    const float wsl = warp_sum(sl > 0.f ? sl * fast_exp2((ml - wml) * l2s) : 0.f);
    const float wsd = warp_sum(sd > 0.f ? sd * fast_exp2((md - wmd) * l2s) : 0.f);
    if (lane == 0) {
      sc.pair[w][0] = wml;
      sc.pair[w][1] = wsl;
      sc.pair[w][2] = wmd;
      sc.pair[w][3] = wsd;
    }
    __syncthreads();
    float Ml = -INFINITY, Md = -INFINITY;
#pragma unroll
    for (int i = 0; i < kNW; ++i) {
      Ml = fmaxf(Ml, sc.pair[i][0]);
      Md = fmaxf(Md, sc.pair[i][2]);
    }
    float Sp = 0.f, Sq = 0.f;
#pragma unroll
    for (int i = 0; i < kNW; ++i) {
      if (sc.pair[i][1] > 0.f) Sp += sc.pair[i][1] * fast_exp2((sc.pair[i][0] - Ml) * l2s);
      if (sc.pair[i][3] > 0.f) Sq += sc.pair[i][3] * fast_exp2((sc.pair[i][2] - Md) * l2s);
    }
    const float scale_l = ml == -INFINITY ? 0.f : fast_exp2((ml - Ml) * l2s) / Sp;
    const float scale_d = (need_draft && md != -INFINITY) ? fast_exp2((md - Md) * l2s) / Sq : 0.f;
#pragma unroll
    for (int e = 0; e < kNodeElems; ++e) {
      const int v = tid + e * kNodeThreads;
      if (v < V) prow[v] *= scale_l;
      q[e] *= scale_d;
    }
    int parity = 0;

    // ---- V2: the children's accept tests, one reduction per rejection
    float c_prev = 0.f, W_prev = 1.f;
    for (int j = 0; j < k; ++j) {
      const int ch = ts.child[j];
      const float P = precise_prob(ts.cP[j], Ml, T_, iT, Sp);
      const float Q = precise_prob(ts.cQ[j], Md, T_, iT, Sq);
      const float alpha = Q > 0.f ? fminf(1.f, fmaxf(0.f, fmaf(-c_prev, Q, P)) / (W_prev * Q)) : 1.f;
      if (tid == 0) {
        const float uu = ts.cU[j];
        int f = (uu < alpha) ? kFlagAccept : 0;
        if (fabsf(uu - alpha) < kTieBand) f |= kFlagTie;
        a.flags[c.lo + ch] = f;
      }
      const float c_new = c_prev + W_prev;
      float ws = 0.f;
#pragma unroll
      for (int e = 0; e < kNodeElems; ++e) {
        const int v = tid + e * kNodeThreads;
        if (v < V) ws += fmaxf(0.f, fmaf(-c_new, q[e], prow[v]));
      }
      const float Wn = node_block_sum(ws, sc, parity);
      parity ^= 1;
      if (Wn > 0.f) {  // otherwise the residual is all zero: keep r
        c_prev = c_new;
        W_prev = Wn;
      }
    }

    // ---- V3: the draw from r ∝ max(0, p - c q) (c = 0: r = p) by inverse CDF
    float total;
    if (c_prev != 0.f) {
#pragma unroll
      for (int e = 0; e < kNodeElems; ++e) {
        const int v = tid + e * kNodeThreads;
        if (v < V) prow[v] = fmaxf(0.f, fmaf(-c_prev, q[e], prow[v]));
      }
    }
    __syncthreads();
    // level 1: one contiguous segment per warp
    const int seg1 = (V + kNW - 1) / kNW;
    const int b1 = min(V, w * seg1), e1 = min(V, b1 + seg1);
    float s1 = 0.f;
    for (int v = b1 + lane; v < e1; v += 32) s1 += prow[v];
    s1 = warp_sum(s1);
    if (lane == 0) sc.lvl[w] = s1;
    __syncthreads();
    total = 0.f;
#pragma unroll
    for (int i = 0; i < kNW; ++i) total += sc.lvl[i];
    const float target = ts.ufb * total;
    float prefix = 0.f;
    bool clamp = false;
    const int w1 = pick_bucket(sc.lvl, kNW, target, prefix, clamp);
    // level 2: that segment in one sub-segment per warp (at most 128 entries)
    const int base2 = w1 * seg1, end2 = min(V, base2 + seg1);
    const int seg2 = (seg1 + kNW - 1) / kNW;
    const int b2 = min(end2, base2 + w * seg2), e2 = min(end2, b2 + seg2);
    float s2 = 0.f;
    for (int v = b2 + lane; v < e2; v += 32) s2 += prow[v];
    s2 = warp_sum(s2);
    __syncthreads();  // every thread has read level 1
    if (lane == 0) sc.lvl[w] = s2;
    __syncthreads();
    const int w2 = pick_bucket(sc.lvl, kNW, target, prefix, clamp);
    // level 3: one warp scans the chosen sub-segment, 32 entries at a time
    if (w == 0) {
      const int b3 = min(end2, base2 + w2 * seg2), e3 = min(end2, b3 + seg2);
      float run = prefix;
      int pick = -1, last_pos = -1;
      float cb0 = target, cb1 = target, last_end = prefix;
      for (int base = b3; base < e3; base += 32) {
        const int v = base + lane;
        const float wv = v < e3 ? prow[v] : 0.f;
        float inc = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const float cum = run + inc;
        const uint32_t pos = __ballot_sync(0xffffffffu, v < e3 && wv > 0.f);
        if (pos) {
          const int L = 31 - __clz(pos);
          last_pos = base + L;
          last_end = __shfl_sync(0xffffffffu, cum, L);
        }
        const uint32_t hit = clamp ? 0u : __ballot_sync(0xffffffffu, v < e3 && cum > target);
        if (hit) {
          const int L = __ffs(hit) - 1;
          pick = base + L;
          cb1 = __shfl_sync(0xffffffffu, cum, L);
          cb0 = cb1 - __shfl_sync(0xffffffffu, wv, L);
          break;
        }
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (pick < 0) {  // not crossed here: the last positive weight of the sub-segment
        clamp = true;
        pick = last_pos >= 0 ? last_pos : b3;
        cb0 = cb1 = last_end;
      }
      if (lane == 0) {
        const bool tie = clamp || fabsf(target - cb0) < kTieBand * total ||
                         fabsf(target - cb1) < kTieBand * total;
        a.fallback[t] = pick | (tie ? (1 << 31) : 0);
      }
    }
  } else if (tid == 0 && c.b >= 0) {
    report(a.status, c.b, c.err);
  }
  __syncthreads();
  arrive_and_walk(a, c, ts, gridDim.x);
}

int launch_verify_node(const VerifyArgs &args, cudaStream_t stream) {
  const bool greedy = !(args.temp > 0.f);
  if (greedy) {
    tree_verify_greedy_node_kernel<<<args.T, kGreedyThreads, 0, stream>>>(args);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  if (args.V > kNodeMaxV) return SPEC_ERR_SHAPE;
  const size_t smem = sizeof(float) * static_cast<size_t>(args.V);
  static int configured = -1;
  if (configured < static_cast<int>(smem)) {
    if (cudaFuncSetAttribute(tree_verify_stoch_node_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SPEC_ERR_CUDA;
    configured = static_cast<int>(smem);
  }
  tree_verify_stoch_node_kernel<<<args.T, kNodeThreads, smem, stream>>>(args);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace spec
