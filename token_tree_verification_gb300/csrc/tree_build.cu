// Draft token-tree construction on the device: one level of expansion and
// the pruning of the candidate tree.
//
// SpecInfer developer article §2.1: the speculator proposes, from each
// node's draft distribution, the candidate tokens that form the next level
// of the token tree, and each node keeps its parent pointer (the deployment
// configuration sets the tree width).
//
// Expansion: one CTA per frontier row.  q = softmax(draft / T), or for T = 0
// the greedy draft (q = softmax(draft), children = its `width` most likely
// tokens, ties to the lower index); T > 0 draws `width` i.i.d. children by
// inverse CDF at the uniforms of counter (node, request, 2, slot).  A child's
// score is its parent's plus log q(token).
// Pruning: one CTA per request; the root and the keep - 1 best other
// candidates by (score desc, index asc) survive, renumbered in order.
#include <algorithm>

#include "common.cuh"

namespace spec {

namespace {

constexpr int kExThreads = 512;
constexpr int kExWarps = kExThreads / 32;
constexpr int kMaxWidth = 16;
constexpr int kExSlice = 8192;   // vocabulary entries per CTA of an expansion cluster
constexpr int kExMaxCS = 8;
constexpr int kPruneThreads = 1024;
constexpr float kDrawTieBand = 1e-6f;

struct ExpandArgs {
  const float *draft, *parent_scores;
  const int32_t *node_ids, *reqs;
  int F, V, width;
  float temp, l2s;   // l2s = log2(e) / T' with T' = T (T > 0) or 1
  uint64_t seed;
  int32_t *tokens, *ties;
  float *scores;
};

struct Cand {   // a candidate token: larger value first, then lower index
  float v;
  int i;
};

__device__ __forceinline__ bool cand_before(Cand a, Cand b) {
  return a.v > b.v || (a.v == b.v && a.i < b.i);
}

__device__ __forceinline__ float wmax(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float wsum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ uint64_t philox_word0(uint64_t seed, uint64_t c0, uint64_t c1, uint64_t c2,
                                                 uint64_t c3) {
  U64x4 c;
  c.w[0] = c0;
  c.w[1] = c1;
  c.w[2] = c2;
  c.w[3] = c3;
  return philox4x64_10(c, seed, 0).w[0];
}

// Expansion of one frontier row by a cluster of CS CTAs, CTA `rank` taking
// the slice [v0, v1) of the vocabulary.  The slices' (max, sum) pairs go to
// every CTA (st.async, completing on each CTA's barrier) and are combined in
// rank order, so every CTA holds the same M and S.  Greedy: each CTA finds its
// slice's best `width` tokens and rank 0 merges the CS lists.  Sampled: each
// CTA scans its slice in contiguous chunks; the slice totals go to every CTA,
// and slice r owns [P_r, P_r + T_r) of [0, S) with P_r = T_0 + ... + T_{r-1}
// added in rank order, so the slices (and the chunks inside them) partition
// [0, S) exactly and each draw is taken by exactly one chunk.
__global__ void __launch_bounds__(kExThreads, 1)
tree_expand_kernel(const ExpandArgs a) {
  __shared__ float s_m[kExWarps], s_s[kExWarps];
  __shared__ Cand s_c[kExWarps];
  __shared__ float s_scan[kExWarps];
  __shared__ float s_pre[kExThreads];   // each chunk's exclusive prefix within the slice
  __shared__ float s_u[kMaxWidth], s_val[kMaxWidth];
  __shared__ int s_tok[kMaxWidth], s_tie[kMaxWidth], s_claim[kMaxWidth];
  __shared__ float s_M, s_S;
  __shared__ __align__(16) float2 x_stat[kExMaxCS];            // every slice's (max, scaled sum)
  __shared__ __align__(16) float x_tot[kExMaxCS];              // every slice's total (sampled)
  __shared__ __align__(16) float2 x_cand[kExMaxCS][kMaxWidth];  // rank 0: every slice's list
  __shared__ __align__(8) uint64_t xbar[2];
  const int CS = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_rank());
  const int f = blockIdx.x / CS, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int V = a.V, W = a.width;
  const bool greedy = !(a.temp > 0.f);
  const int slice = (V + CS - 1) / CS;
  const int v0 = min(V, rank * slice), v1 = min(V, v0 + slice);
  if (tid == 0) {
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&xbar[0], static_cast<uint32_t>(CS * 8));
    if (!greedy) mbar_arrive_expect_tx(&xbar[1], static_cast<uint32_t>(CS * 4));
    else if (rank == 0) mbar_arrive_expect_tx(&xbar[1], static_cast<uint32_t>(CS * W * 8));
  }
  cluster_arrive_relaxed();   // barriers initialised; waited for before the first remote store
  pdl_trigger();
  pdl_wait();
  const float *row = a.draft + static_cast<size_t>(f) * V;
  bool ok = true;

  // ---- pass A over the slice: max and sum of 2^((x - max) * l2s); the
  //      greedy draft also keeps each thread's best `width` candidates
  Cand best[kMaxWidth];
#pragma unroll
  for (int j = 0; j < kMaxWidth; ++j) best[j] = Cand{-INFINITY, 0x7fffffff};
  // greedy: strided over the slice; sampled: over this thread's contiguous
  // chunk of the slice, whose (max, sum) then also gives the chunk's mass
  const int len = v1 - v0;
  const int C = (len + kExThreads - 1) / kExThreads;
  const int c0 = v0 + min(len, tid * C), c1 = v0 + min(len, tid * C + C);
  const int xs = greedy ? v0 + tid : c0, xe = greedy ? v1 : c1, xd = greedy ? kExThreads : 1;
  float m = -INFINITY, s = 0.f;
  for (int x = xs; x < xe; x += xd) {
    const float v = __ldg(row + x);
    if (v > m) {
      s = (m == -INFINITY ? 0.f : s * fast_exp2((m - v) * a.l2s)) + 1.f;
      m = v;
    } else if (m != -INFINITY) {   // a -inf logit before any finite one adds nothing
      s += fast_exp2((v - m) * a.l2s);
    }
    if (greedy) {
      Cand c{v, x};
#pragma unroll
      for (int j = 0; j < kMaxWidth; ++j) {   // insertion into the sorted list
        if (j < W && cand_before(c, best[j])) {
          const Cand t = best[j];
          best[j] = c;
          c = t;
        }
      }
    }
  }
  {
    float wm = wmax(m);
    float ws = s > 0.f ? s * fast_exp2((m - wm) * a.l2s) : 0.f;
    ws = wsum(ws);
    if (lane == 0) {
      s_m[w] = wm;
      s_s[w] = ws;
    }
    __syncthreads();
    if (w == 0) {
      const float pm = lane < kExWarps ? s_m[lane] : -INFINITY;
      const float ps = lane < kExWarps ? s_s[lane] : 0.f;
      const float Mr = wmax(pm);
      const float Sr = wsum(ps > 0.f ? ps * fast_exp2((pm - Mr) * a.l2s) : 0.f);
      cluster_wait();
      if (lane < CS)
        st_async_v2_f32(peer_addr(&x_stat[rank], lane), Mr, Sr, peer_addr(&xbar[0], lane));
    } else {
      cluster_wait();
    }
    if (!mbar_wait(&xbar[0], 0)) ok = false;
    float M = -INFINITY;
    for (int q = 0; q < CS; ++q) M = fmaxf(M, x_stat[q].x);
    float S = 0.f;
    for (int q = 0; q < CS; ++q)
      if (x_stat[q].y > 0.f) S += x_stat[q].y * fast_exp2((x_stat[q].x - M) * a.l2s);
    if (tid == 0) {
      s_M = M;
      s_S = S;
    }
    __syncthreads();
  }
  const float M = s_M;

  if (greedy) {
    // ---- the slice's best `width`: rounds of a block-wide argmax over the
    //      threads' list heads
    int head = 0;
    for (int j = 0; j < W; ++j) {
      Cand c = head < W ? best[0] : Cand{-INFINITY, 0x7fffffff};
#pragma unroll
      for (int k = 1; k < kMaxWidth; ++k)
        if (k == head && k < W) c = best[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const Cand y{__shfl_xor_sync(0xffffffffu, c.v, o), __shfl_xor_sync(0xffffffffu, c.i, o)};
        if (cand_before(y, c)) c = y;
      }
      if (lane == 0) s_c[w] = c;
      __syncthreads();
      if (w == 0) {
        Cand b = lane < kExWarps ? s_c[lane] : Cand{-INFINITY, 0x7fffffff};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const Cand y{__shfl_xor_sync(0xffffffffu, b.v, o), __shfl_xor_sync(0xffffffffu, b.i, o)};
          if (cand_before(y, b)) b = y;
        }
        if (lane == 0) {
          s_tok[j] = b.i;
          s_val[j] = b.v;
        }
      }
      __syncthreads();
      // the owner of the winner (token x belongs to thread (x - v0) % threads) pops it
      const int x = s_tok[j];
      if (x >= v0 && x < v1 && (x - v0) % kExThreads == tid) ++head;
    }
    // ---- rank 0 merges the CS lists
    if (tid < W)
      st_async_v2_f32(peer_addr(&x_cand[rank][tid], 0), s_val[tid], __int_as_float(s_tok[tid]),
                      peer_addr(&xbar[1], 0));
    if (rank == 0) {
      if (!mbar_wait(&xbar[1], 0)) ok = false;
      if (w == 0) {
        Cand c[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = lane + 32 * k;   // candidate e: list e / W, entry e % W
          c[k] = e < CS * W ? Cand{x_cand[e / W][e % W].x, __float_as_int(x_cand[e / W][e % W].y)}
                            : Cand{-INFINITY, 0x7fffffff};
        }
        for (int j = 0; j < W; ++j) {
          Cand b = c[0];
          int kb = 0;
#pragma unroll
          for (int k = 1; k < 4; ++k)
            if (cand_before(c[k], b)) {
              b = c[k];
              kb = k;
            }
          Cand g = b;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const Cand y{__shfl_xor_sync(0xffffffffu, g.v, o), __shfl_xor_sync(0xffffffffu, g.i, o)};
            if (cand_before(y, g)) g = y;
          }
          if (b.i == g.i && b.v == g.v) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k == kb) c[k] = Cand{-INFINITY, 0x7fffffff};   // the winner leaves its lane
          }
          if (lane == 0) {
            const int x = min(max(g.i, 0), V - 1);
            const float lq = (g.v - M) * (a.l2s * 0.6931471805599453f) - logf(s_S);
            a.tokens[static_cast<size_t>(f) * W + j] = x;
            a.scores[static_cast<size_t>(f) * W + j] = __ldg(a.parent_scores + f) + lq;
            a.ties[static_cast<size_t>(f) * W + j] = ok ? 0 : -1;
          }
        }
      }
    }
  } else {
    // ---- inverse CDF: contiguous chunks of the slice, exclusive scan of chunk
    //      sums (a chunk's sum from its own (max, sum) of pass A)
    const float cs = s > 0.f ? s * fast_exp2((m - M) * a.l2s) : 0.f;
    float inc = cs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) s_scan[w] = inc;
    if (tid < W) {
      const uint64_t word = philox_word0(a.seed, static_cast<uint64_t>(__ldg(a.node_ids + f)),
                                         static_cast<uint64_t>(__ldg(a.reqs + f)), 2,
                                         static_cast<uint64_t>(tid));
      s_u[tid] = static_cast<float>(word >> 40) * (1.0f / 16777216.0f);
      s_claim[tid] = 0;
    }
    __syncthreads();
    if (w == 0) {
      const float v = lane < kExWarps ? s_scan[lane] : 0.f;
      float x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane < kExWarps) s_scan[lane] = x - v;   // exclusive prefix of the warps
      const float T = __shfl_sync(0xffffffffu, x, kExWarps - 1);   // the slice's total
      if (lane < CS) st_async_f32(peer_addr(&x_tot[rank], lane), T, peer_addr(&xbar[1], lane));
    }
    __syncthreads();
    const float pre = s_scan[w] + inc - cs;
    s_pre[tid] = pre;
    if (!mbar_wait(&xbar[1], 0)) ok = false;
    // the slices' offsets and the row's total, added in rank order
    float P = 0.f, S = 0.f;
    for (int q = 0; q < CS; ++q) {
      if (q == rank) P = S;
      S += x_tot[q];
    }
    const float T = x_tot[rank];
    __syncthreads();
    if (tid == 0) s_S = S;
    // chunk t owns [P + pre_t, P + pre_{t+1}), the last one up to P + T
    const float begin = P + pre;
    const float end = P + (tid + 1 < kExThreads ? s_pre[tid + 1] : T);
    for (int j = 0; j < W; ++j) {
      const float target = s_u[j] * S;
      const bool last_chunk = rank == CS - 1 && tid == kExThreads - 1;
      if (begin <= target && (target < end || (last_chunk && target >= end))) {
        float run = begin;
        int pick = -1;
        float cb0 = target, cb1 = target;
        for (int x = c0; x < c1 && pick < 0; ++x) {
          const float e = fast_exp2((__ldg(row + x) - M) * a.l2s);
          if (run + e > target) {
            pick = x;
            cb0 = run;
            cb1 = run + e;
          }
          run += e;
        }
        if (pick < 0) {  // rounding: the chunk's last entry of positive weight, on the boundary
          for (int x = c1 - 1; x >= c0 && pick < 0; --x)
            if (fast_exp2((__ldg(row + x) - M) * a.l2s) > 0.f) pick = x;
          if (pick < 0) pick = max(c0, min(V - 1, c1 - 1));
          cb0 = cb1 = target;
        }
        s_tok[j] = pick;
        s_tie[j] = fabsf(target - cb0) < kDrawTieBand * S || fabsf(target - cb1) < kDrawTieBand * S;
        s_claim[j] = 1;
      }
    }
    __syncthreads();
    if (tid < W && s_claim[tid]) {
      const int x = min(max(s_tok[tid], 0), V - 1);   // in range for any row contents
      const float lq = (__ldg(row + x) - M) * (a.l2s * 0.6931471805599453f) - logf(S);
      a.tokens[static_cast<size_t>(f) * W + tid] = x;
      a.scores[static_cast<size_t>(f) * W + tid] = __ldg(a.parent_scores + f) + lq;
      a.ties[static_cast<size_t>(f) * W + tid] = ok ? s_tie[tid] : -1;
    }
  }
}

struct PruneArgs {
  const int32_t *parents, *tokens, *offsets;
  const float *scores;
  int B, keep;
  int32_t *out_parents, *out_tokens, *kept, *n_out, *status;
};

__global__ void __launch_bounds__(kPruneThreads)
tree_prune_kernel(const PruneArgs a) {
  __shared__ float sc[kPruneThreads];
  __shared__ int par[kPruneThreads], newid[kPruneThreads], wsum[kPruneThreads / 32];
  __shared__ int s_bad;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  pdl_trigger();
  pdl_wait();
  const int lo = __ldg(a.offsets + b), n = __ldg(a.offsets + b + 1) - lo;
  int32_t *op = a.out_parents + static_cast<size_t>(b) * a.keep;
  int32_t *ot = a.out_tokens + static_cast<size_t>(b) * a.keep;
  int32_t *ok_ = a.kept + static_cast<size_t>(b) * a.keep;
  for (int i = tid; i < a.keep; i += kPruneThreads) {
    op[i] = -2;
    ot[i] = -1;
    ok_[i] = -1;
  }
  if (n < 1 || n > kPruneThreads) {
    if (tid == 0) {
      report(a.status, b, SPEC_ERR_TREE_TOO_LARGE);
      a.n_out[b] = 0;
    }
    return;
  }
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (tid < n) {
    // (the candidate arrays hold cand_offsets[B] entries)
    const bool in = in_bounds(lo + tid, kChecked ? __ldg(a.offsets + a.B) : 0, a.status, b);
    const int p = in ? __ldg(a.parents + lo + tid) : -2;
    par[tid] = p;
    sc[tid] = in ? __ldg(a.scores + lo + tid) : -INFINITY;
    if (tid == 0 ? p != -1 : (p < 0 || p >= tid)) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      report(a.status, b, SPEC_ERR_BAD_PARENT);
      a.n_out[b] = 0;
    }
    return;
  }
  // rank among the non-root candidates: (score desc, index asc)
  bool keep_me = tid == 0;
  if (tid >= 1 && tid < n) {
    const float si = sc[tid];
    int better = 0;
    for (int j = 1; j < n; ++j) {
      const float sj = sc[j];
      better += (sj > si || (sj == si && j < tid)) ? 1 : 0;
    }
    keep_me = better < a.keep - 1;
  }
  // new index = number of kept candidates before this one
  const unsigned bal = __ballot_sync(0xffffffffu, keep_me);
  if (lane == 0) wsum[w] = __popc(bal);
  __syncthreads();
  int before = __popc(bal & ((1u << lane) - 1u));
  for (int k = 0; k < w; ++k) before += wsum[k];
  newid[tid] = keep_me ? before : -1;
  __syncthreads();
  if (keep_me && tid < n && in_bounds(before, a.keep, a.status, b)) {
    op[before] = tid == 0 ? -1 : newid[par[tid]];
    ot[before] = __ldg(a.tokens + lo + tid);
    ok_[before] = tid;
  }
  if (tid == kPruneThreads - 1) {
    int total = 0;
    for (int k = 0; k < kPruneThreads / 32; ++k) total += wsum[k];
    a.n_out[b] = total;
  }
}

}  // namespace

}  // namespace spec

extern "C" int spec_tree_expand(const float *draft_logits, const float *parent_scores,
                                const int32_t *node_ids, const int32_t *requests, int F, int V,
                                int width, float temperature, uint64_t seed, int32_t *child_tokens,
                                float *child_scores, int32_t *near_ties, void *stream) {
  using namespace spec;
  if (!draft_logits || !parent_scores || !node_ids || !requests || !child_tokens || !child_scores ||
      !near_ties)
    return SPEC_ERR_NULL;
  if (F < 1 || V < 1 || width < 1 || width > kMaxWidth || width > V) return SPEC_ERR_SHAPE;
  if (!(temperature >= 0.f) || temperature > 1e4f) return SPEC_ERR_SHAPE;
  ExpandArgs args;
  args.draft = draft_logits;
  args.parent_scores = parent_scores;
  args.node_ids = node_ids;
  args.reqs = requests;
  args.F = F;
  args.V = V;
  args.width = width;
  args.temp = temperature;
  args.l2s = 1.4426950408889634f / (temperature > 0.f ? temperature : 1.f);
  args.seed = seed;
  args.tokens = child_tokens;
  args.scores = child_scores;
  args.ties = near_ties;
  const int CS = std::min(kExMaxCS, (V + kExSlice - 1) / kExSlice);   // CTAs per row
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(F) * CS, 1, 1);
  cfg.blockDim = dim3(kExThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attribute(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tree_expand_kernel, args) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_tree_prune(const int32_t *parents, const int32_t *tokens, const float *scores,
                               const int32_t *cand_offsets, int B, int keep, int32_t *out_parents,
                               int32_t *out_tokens, int32_t *kept_index, int32_t *n_out,
                               int32_t *status, void *stream) {
  using namespace spec;
  if (!parents || !tokens || !scores || !cand_offsets || !out_parents || !out_tokens || !kept_index ||
      !n_out || !status)
    return SPEC_ERR_NULL;
  if (B < 1 || keep < 1 || keep > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  PruneArgs args;
  args.parents = parents;
  args.tokens = tokens;
  args.offsets = cand_offsets;
  args.scores = scores;
  args.B = B;
  args.keep = keep;
  args.out_parents = out_parents;
  args.out_tokens = out_tokens;
  args.kept = kept_index;
  args.n_out = n_out;
  args.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(kPruneThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  pdl_attribute(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_prune_kernel, args) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
