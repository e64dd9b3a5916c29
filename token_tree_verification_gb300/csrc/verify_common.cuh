// Pieces shared by the two verification kernels (one thread-block cluster
// per node for large vocabularies, one CTA per node otherwise): arguments,
// reductions, the accept-ratio helper, loading a node's tree context, and the
// per-request arrival that runs the root-to-leaf walk.
//
// Sources: speculative-decoding explainer (intelliparadigm.com) §2.2
// 三阶段工作流程详解 (stage 2: alpha = min(1, p/q); stage 3: stop at the first
// rejection and draw a new target prediction); SpecInfer developer article
// §2.1 (accept the longest verified prefix).
#pragma once

#include "common.cuh"

namespace spec {

constexpr int kVThreads = 1024;    // cluster kernel: threads per CTA
constexpr int kVWarps = kVThreads / 32;
constexpr int kMaxCS = 8;          // CTAs per cluster (portable limit)
constexpr int kChunkTarget = 16384;  // vocabulary entries per CTA the cluster size aims at
constexpr int kMaxChunk = 27648;   // floats per CTA per row (2 rows fit in 216 KB)
constexpr int kGreedyThreads = 1024;  // greedy per-node kernel: threads per CTA
constexpr int kTreeWindow = 2 * SPEC_MAX_TREE_NODES - 1;   // nodes t-127 .. t+127
constexpr int kFlagAccept = 1;
constexpr int kFlagTie = 2;
constexpr float kTieBand = 1e-6f;

struct VerifyArgs {
  const float *target;
  const float *draft;
  const int32_t *tokens;
  const int32_t *parents;
  const int32_t *offsets;
  int B, T, V, chunk, W;
  float temp;     // 0 => greedy
  float inv_temp;
  uint64_t seed;
  int32_t *accept_len, *path_nodes, *out_tokens, *near_ties, *status;
  int32_t *flags;      // [T] written by the parent's CTA group: accept / tie bits
  int32_t *fallback;   // [T] token emitted on stopping at the node | tie << 31
  uint32_t *done;      // [B] arrival counters, then one global counter at [B]
};

// A node's tree context, staged in shared memory by load_tree().
struct TreeSmem {
  int wpar[kTreeWindow + 1];          // parents / tokens of nodes t-127 .. t+127
  int wtok[kTreeWindow + 1];
  int par[SPEC_MAX_TREE_NODES];
  int tok[SPEC_MAX_TREE_NODES];
  int child[SPEC_MAX_TREE_NODES];     // u's children in index order
  float cP[SPEC_MAX_TREE_NODES];      // target logit of each child's token
  float cQ[SPEC_MAX_TREE_NODES];      // draft logit of each child's token
  float cU[SPEC_MAX_TREE_NODES];      // the accept-test uniform of each child
  int warp_cnt[SPEC_MAX_TREE_NODES / 32];
  int meta[4];                        // error, request
  float ufb;                          // the uniform of u's fallback draw
  int walk;
};

struct NodeCtx {
  int b, lo, n, u, k, err;
};

// ---------------------------------------------------------------- reductions
struct ArgMax {
  float v;
  int i;
};

__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
  // larger value wins; equal values: lower index wins
  return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = better(a, b);
  }
  return a;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}




// p(x) = exp((l - M) / temp) / S with the exponent's argument carried to
// near double precision (TwoSum for l - M, an FMA remainder for the
// division), so the accept ratio is as accurate as fp32 exp allows.
__device__ __forceinline__ float precise_prob(float l, float M, float temp, float inv_temp,
                                              float S) {
  const float d_hi = l - M;
  const float bv = d_hi - l;
  const float d_lo = (l - (d_hi - bv)) + (-M - bv);
  const float z_hi = d_hi * inv_temp;
  const float rem = fmaf(-z_hi, temp, d_hi);
  const float z_lo = (rem + d_lo) * inv_temp;
  const float e = expf(z_hi);
  return fmaf(e, z_lo, e) / S;
}

// ---------------------------------------------------------------- the walk
// One warp walks request b from the root (step V4).  Node i's data sits in
// lane i % 32, slot i / 32.
// spar / stok: the request's parents and tokens, staged in shared memory.
static __device__ void walk_request(const VerifyArgs &a, int b, int lo, int n, const int *spar,
                             const int *stok) {
  const int lane = threadIdx.x & 31;
  if (*reinterpret_cast<volatile int32_t *>(a.status + b) != 0) return;
  int par[4], flg[4], fbk[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int i = lane + 32 * s;
    par[s] = i < n ? spar[i] : -2;
    flg[s] = i < n ? __ldcg(a.flags + lo + i) : 0;
    fbk[s] = i < n ? __ldcg(a.fallback + lo + i) : 0;
  }
  // depth of each node (parents are validated: parent < index)
  int maxd = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int i = lane + 32 * s;
    if (i < n) {
      int d = 0;
      for (int x = i; x > 0; x = spar[x]) ++d;
      maxd = max(maxd, d);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxd = max(maxd, __shfl_xor_sync(0xffffffffu, maxd, o));
  if (maxd + 1 > a.W) {
    if (lane == 0) report(a.status, b, SPEC_ERR_TREE_TOO_LARGE);
    return;
  }
  int32_t *pn = a.path_nodes + static_cast<size_t>(b) * a.W;
  int32_t *ot = a.out_tokens + static_cast<size_t>(b) * a.W;
  int cur = 0, acc = 0, ties = 0;
  for (;;) {
    int next = -1;
    uint32_t tie_bits[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const bool child = par[s] == cur;
      tie_bits[s] = __ballot_sync(0xffffffffu, child && (flg[s] & kFlagTie));
      const uint32_t ok = __ballot_sync(0xffffffffu, child && (flg[s] & kFlagAccept));
      if (next < 0 && ok) next = 32 * s + __ffs(ok) - 1;
    }
    // decisions taken at this node: children up to and including `next`
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t m = tie_bits[s];
      if (next >= 0) {
        const int lim = next - 32 * s;  // keep bits <= lim
        m = lim < 0 ? 0u : (lim >= 31 ? m : (m & ((2u << lim) - 1u)));
      }
      ties += __popc(m);
    }
    if (next < 0) {
      // the fallback of node `cur` sits in lane cur % 32, slot cur / 32
      const int f0 = __shfl_sync(0xffffffffu, fbk[0], cur & 31);
      const int f1 = __shfl_sync(0xffffffffu, fbk[1], cur & 31);
      const int f2 = __shfl_sync(0xffffffffu, fbk[2], cur & 31);
      const int f3 = __shfl_sync(0xffffffffu, fbk[3], cur & 31);
      const int sl = cur >> 5;
      const int fb = sl == 0 ? f0 : (sl == 1 ? f1 : (sl == 2 ? f2 : f3));
      if (lane == 0) ot[acc] = fb & 0x7fffffff;
      ties += (fb >> 31) & 1;
      break;
    }
    if (lane == 0) {
      ot[acc] = stok[next];
      pn[acc + 1] = next;
    }
    ++acc;
    cur = next;
  }
  if (lane == 0) {
    pn[0] = 0;
    for (int j = acc + 1; j < a.W; ++j) {
      pn[j] = -1;
      ot[j] = -1;
    }
    a.accept_len[b] = acc;
    a.near_ties[b] = ties;
  }
}

// ---------------------------------------------------------------- kernel
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}


// Every thread of the CTA (blockDim >= 256) calls this: find node t's
// request, stage its parents and tokens, validate them, and list u's
// children in index order.  Errors are identical in every CTA of a group.
// A request holds at most 128 nodes, so the parents and tokens of nodes
// t-127 .. t+127 are loaded in the same round as the offsets.
static __device__ NodeCtx load_tree(const VerifyArgs &a, int t, TreeSmem &ts) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    ts.meta[0] = 0;
    ts.meta[1] = -1;
  }
  if (tid < kTreeWindow) {
    const int x = t - (SPEC_MAX_TREE_NODES - 1) + tid;
    const bool in = x >= 0 && x < a.T;
    ts.wpar[tid] = in ? __ldg(a.parents + x) : -2;
    ts.wtok[tid] = in ? __ldg(a.tokens + x) : 0;
  }
  __syncthreads();
  if (a.B < static_cast<int>(blockDim.x)) {
    if (tid < a.B) {
      const int o0 = __ldg(a.offsets + tid), o1 = __ldg(a.offsets + tid + 1);
      if (o0 <= t && t < o1) atomicMax(&ts.meta[1], tid);
    }
  } else if (tid == 0) {
    ts.meta[1] = find_request(a.offsets, a.B, t);
  }
  __syncthreads();
  NodeCtx c;
  c.b = ts.meta[1];
  c.lo = c.n = c.k = 0;
  c.err = 0;
  if (c.b < 0) {
    c.err = SPEC_ERR_TREE_TOO_LARGE;
  } else {
    c.lo = __ldg(a.offsets + c.b);
    c.n = __ldg(a.offsets + c.b + 1) - c.lo;
    if (c.lo < 0 || c.lo + c.n > a.T || c.n < 1 || c.n > SPEC_MAX_TREE_NODES)
      c.err = SPEC_ERR_TREE_TOO_LARGE;
  }
  c.u = t - c.lo;
  bool is_child = false;
  uint32_t child_bal = 0;
  if (!c.err && tid < SPEC_MAX_TREE_NODES) {
    if (tid < c.n) {
      const int wi = c.lo + tid - (t - (SPEC_MAX_TREE_NODES - 1));   // in [0, 254]
      const int p = ts.wpar[wi];
      const int x = ts.wtok[wi];
      ts.par[tid] = p;
      ts.tok[tid] = x;
      const bool ok = (tid == 0) ? (p == -1) : (p >= 0 && p < tid);
      if (!ok) atomicCAS(&ts.meta[0], 0, SPEC_ERR_BAD_PARENT);
      is_child = (tid > c.u && p == c.u);
      if (is_child && (x < 0 || x >= a.V)) atomicCAS(&ts.meta[0], 0, SPEC_ERR_TOKEN_RANGE);
    }
    child_bal = __ballot_sync(0xffffffffu, is_child);
    if (lane == 0) ts.warp_cnt[w] = __popc(child_bal);
  }
  __syncthreads();
  if (!c.err) c.err = ts.meta[0];
  if (!c.err) {
    int before = 0;
    for (int i = 0; i < SPEC_MAX_TREE_NODES / 32; ++i) {
      if (i < w) before += ts.warp_cnt[i];
      c.k += ts.warp_cnt[i];
    }
    if (is_child) ts.child[before + __popc(child_bal & ((1u << lane) - 1u))] = tid;
  }
  __syncthreads();  // child list complete
  return c;
}

// Uniforms of the children's accept tests and of u's fallback draw, and the
// children's logits at their tokens (stochastic mode), in parallel.
__device__ __forceinline__ void load_children(const VerifyArgs &a, const NodeCtx &c, int t,
                                              TreeSmem &ts) {
  const int tid = threadIdx.x;
  if (c.err || !(a.temp > 0.f)) return;
  const float *trow = a.target + static_cast<size_t>(t) * a.V;
  const float *drow = a.draft + static_cast<size_t>(t) * a.V;
  if (tid < c.k) {
    const int ch = ts.child[tid];
    const int x = ts.tok[ch];
    ts.cP[tid] = __ldg(trow + x);
    ts.cQ[tid] = __ldg(drow + x);
    ts.cU[tid] = spec_uniform(a.seed, ch, c.b, 0);
  } else if (tid == static_cast<int>(blockDim.x) - 1) {
    ts.ufb = spec_uniform(a.seed, c.u, c.b, 1);
  }
}

// Called by every thread of one CTA per node group once the group's outputs
// are written: the last group of a request walks it, and the last group of
// the grid clears every counter for the next call.
static __device__ void arrive_and_walk(const VerifyArgs &a, const NodeCtx &c, TreeSmem &ts, int ngroups) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    __threadfence();
    int walk = 0;
    if (c.b >= 0) {
      const uint32_t prev = atomicAdd(a.done + c.b, 1u);
      walk = (!c.err && static_cast<int>(prev) == c.n - 1) ? 1 : 0;
    }
    ts.walk = walk;
  }
  __syncthreads();
  if (ts.walk) {
    __threadfence();
    if (tid < 32) walk_request(a, c.b, c.lo, c.n, ts.par, ts.tok);
  }
  if (tid == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(a.done + a.B, 1u);
    if (static_cast<int>(prev) == ngroups - 1)
      for (int i = 0; i <= a.B; ++i) a.done[i] = 0u;
  }
}

// greedy per-node kernel (verify_node.cu)
int launch_verify_greedy(const VerifyArgs &args, cudaStream_t stream);

}  // namespace spec
