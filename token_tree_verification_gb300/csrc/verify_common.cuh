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
  float top_p;    // nucleus mass (1: no filter)
  uint64_t seed;
  int32_t *accept_len, *path_nodes, *out_tokens, *near_ties, *status;
  int32_t *flags;      // [T] written by the parent's CTA group: accept / tie bits
  int32_t *fallback;   // [T] token emitted on stopping at the node | tie << 31
  uint32_t *done;      // [B] arrival counters (zero between calls)
  uint64_t wait_ns;    // limit of every bounded wait (kWaitLimitNs outside the failure test)
  int drop_request;    // failure test: this request's first exchange is withheld (-1: none)
  int prefetch_rows;   // stochastic kernel: every node prefetches its target slice into L2
                       // at once (set when all the launch's CTAs are resident together)
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
  int wmatch[32];                     // per warp: the request found to own the node, or -1
  int wbad[32];                       // per warp: the offsets break their contract
  int meta[4];                        // error, child count, first node, node count
  float ufb;                          // the uniform of u's fallback draw
  int walk;
  int stop_fb;                        // the node's fallback token | tie << 31, in the writer CTA
  int timeout;                        // a bounded wait of this CTA ran out
  int fits;                           // the root: the deepest path fits the output rows
  float dm[32], ds[32];               // per warp: (max, sum) of a leaf's row (draw at a leaf)
  int leaf[5];                        // walk ended at a leaf: node, request-local; accepted
                                      // tokens; near-ties so far; the draw's selected range;
                                      // the draw's token | tie << 31
};

struct NodeCtx {
  int b, lo, n, u, k, err;
  bool count;   // the node counts toward its request's arrivals (the offsets are valid)
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

// the warp's maximum (a NaN lane is ignored, as fmaxf does), one reduction
// instruction
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
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
// Arrival word of a request (one u32 per request in the workspace): bits
// 0-15 count the nodes that arrived, bits 16-23 the nodes whose bounded waits
// ran out, bit 24 says the walk ended at the root and the root's CTA wrote
// the request's outputs.
constexpr uint32_t kArriveCount = 0xffffu;
constexpr uint32_t kArriveErr = 1u << 16;
constexpr uint32_t kArriveErrMask = 0xffu << 16;
constexpr uint32_t kArriveRootDone = 1u << 24;

// Whether request b's output rows hold its deepest path (one warp; spar:
// the request's parents, staged in shared memory, already validated).
// path_fits_quiet only answers; path_fits also reports
// SPEC_ERR_TREE_TOO_LARGE when they do not.
static __device__ bool path_fits_quiet(const VerifyArgs &a, int n, const int *spar) {
  const int lane = threadIdx.x & 31;
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
  return maxd + 1 <= a.W;
}

static __device__ bool path_fits(const VerifyArgs &a, int b, int n, const int *spar) {
  const bool fits = path_fits_quiet(a, n, spar);
  if (!fits && (threadIdx.x & 31) == 0) report(a.status, b, SPEC_ERR_TREE_TOO_LARGE);
  return fits;
}

// Outputs of request b when the walk ends at the root without accepting a
// child (one warp): the emitted token alone.
static __device__ void write_root_stop(const VerifyArgs &a, int b, int token, int ties) {
  const int lane = threadIdx.x & 31;
  int32_t *pn = a.path_nodes + static_cast<size_t>(b) * a.W;
  int32_t *ot = a.out_tokens + static_cast<size_t>(b) * a.W;
  for (int j = lane; j < a.W; j += 32) {
    pn[j] = j == 0 ? 0 : -1;
    ot[j] = j == 0 ? token : -1;
  }
  if (lane == 0) {
    a.accept_len[b] = 0;
    a.near_ties[b] = ties;
  }
}

// One warp walks request b from the root (step V4).  Node i's data sits in
// lane i % 32, slot i / 32.
// spar / stok: the request's parents and tokens, staged in shared memory.
// With `lazy_leaves` the leaves computed no fallback: when the walk stops at
// a leaf, the walk records it in ts.leaf (node, accepted count, near-ties)
// and leaves the emitted token and the near-tie count to the caller's draw;
// returns whether it did.
static __device__ bool walk_request(const VerifyArgs &a, int b, int lo, int n, const int *spar,
                                    const int *stok, bool lazy_leaves, TreeSmem &ts) {
  const int lane = threadIdx.x & 31;
  // the request's flags and fallbacks, all in one round trip
  int par[4], flg[4], fbk[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int i = lane + 32 * s;
    par[s] = i < n ? spar[i] : -2;
    const bool in = i < n && in_bounds(lo + i, a.T, a.status, b);
    flg[s] = in ? __ldcg(a.flags + lo + i) : 0;
    fbk[s] = in ? __ldcg(a.fallback + lo + i) : 0;
  }
  if (!path_fits(a, b, n, spar)) return false;
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
    if (next < 0 && lazy_leaves) {
      bool has_child = false;
#pragma unroll
      for (int s = 0; s < 4; ++s) has_child |= __any_sync(0xffffffffu, par[s] == cur);
      if (!has_child) {
        // a leaf: its draw is computed now, by the whole CTA
        if (lane == 0) {
          pn[0] = 0;
          for (int j = acc + 1; j < a.W; ++j) {
            pn[j] = -1;
            ot[j] = -1;
          }
          a.accept_len[b] = acc;
          ts.leaf[0] = cur;
          ts.leaf[1] = acc;
          ts.leaf[2] = ties;
        }
        return true;
      }
    }
    if (next < 0) {
      // the fallback of node `cur` sits in lane cur % 32, slot cur / 32
      const int f0 = __shfl_sync(0xffffffffu, fbk[0], cur & 31);
      const int f1 = __shfl_sync(0xffffffffu, fbk[1], cur & 31);
      const int f2 = __shfl_sync(0xffffffffu, fbk[2], cur & 31);
      const int f3 = __shfl_sync(0xffffffffu, fbk[3], cur & 31);
      const int sl = cur >> 5;
      const int fb = sl == 0 ? f0 : (sl == 1 ? f1 : (sl == 2 ? f2 : f3));
      if (lane == 0 && in_bounds(acc, a.W, a.status, b)) ot[acc] = fb & 0x7fffffff;
      ties += (fb >> 31) & 1;
      break;
    }
    if (lane == 0 && in_bounds(acc + 1, a.W, a.status, b)) {
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
  return false;
}

// The token drawn at a leaf u (the bonus token when the walk accepts the
// path down to it): the inverse-CDF draw from p_u = softmax(row / T) at the
// uniform `u`, taken by the whole CTA (blockDim.x threads, a multiple of 32,
// at most 1024).  Warp w owns the contiguous range [w R, (w + 1) R) of the
// row: one pass gives each warp's (max, sum), the CTA adds the warps'
// masses in index order and finds the range where the running mass passes
// u * S; that range's warp splits it over its lanes, finds the lane's
// stretch, and that lane walks its entries.  Returns token | tie << 31, tie
// when u * S lies within 1e-6 * S of the chosen entry's interval ends; when
// rounding keeps the running sum below u * S, the last entry of positive
// weight (a tie).  Called by every thread; the result is valid in thread 0.
static __device__ int cta_leaf_draw(const float *row, int V, float l2s, float u, TreeSmem &ts) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  const int R = (V + nw - 1) / nw;
  const int r0 = min(V, w * R), r1 = min(V, r0 + R);
  // pass 1: the warp's online (max, sum), lanes strided for coalescing
  float m = -INFINITY, sum = 0.f;
  for (int x = r0 + lane; x < r1; x += 32) {
    const float v = __ldcg(row + x) * l2s;
    if (v > m) {
      sum = sum * fast_exp2(m - v) + 1.f;
      m = v;
    } else if (v != -INFINITY) {
      sum += fast_exp2(v - m);
    }
  }
  const float wm = warp_max(m);
  sum = (m == -INFINITY) ? 0.f : sum * fast_exp2(m - wm);
  sum = warp_sum(sum);
  if (lane == 0) {
    ts.dm[w] = wm;
    ts.ds[w] = sum;
  }
  __syncthreads();
  // the warps' masses relative to the row's max, and where u * S falls
  if (w == 0) {
    const float mw = lane < nw ? ts.dm[lane] : -INFINITY;
    const float M = warp_max(mw);
    const float mass = (lane < nw && ts.ds[lane] > 0.f) ? ts.ds[lane] * fast_exp2(mw - M) : 0.f;
    float inc = mass;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const float S = __shfl_sync(0xffffffffu, inc, 31);
    const float target = u * S;
    const uint32_t hit = __ballot_sync(0xffffffffu, lane < nw && inc > target);
    const uint32_t pos = __ballot_sync(0xffffffffu, mass > 0.f);
    const int ws = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    const float before = __shfl_sync(0xffffffffu, inc - mass, ws);   // mass before warp ws
    if (lane == 0) {
      ts.leaf[3] = ws | (hit ? 0 : (1 << 30));       // bit 30: rounding, no crossing
      ts.dm[0] = M;
      ts.ds[0] = S;
      ts.ds[1] = before;
    }
  }
  __syncthreads();
  const int sel = ts.leaf[3];
  const int ws = sel & 0xffff;
  const bool rounding = (sel >> 30) & 1;
  const float M = ts.dm[0], S = ts.ds[0], before = ts.ds[1];
  const float target = u * S;
  int result = 0;
  if (w == ws) {
    // pass 2: the selected range split into one stretch per lane
    const int a0 = min(V, ws * R), a1 = min(V, a0 + R);
    const int per = (a1 - a0 + 31) / 32;
    const int s0 = min(a1, a0 + lane * per), s1 = min(a1, s0 + per);
    float ls = 0.f;
    for (int x = s0; x < s1; ++x) ls += fast_exp2(__ldcg(row + x) * l2s - M);
    float inc = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t hit = rounding ? 0u : __ballot_sync(0xffffffffu, before + inc > target);
    const uint32_t pos = __ballot_sync(0xffffffffu, ls > 0.f);
    const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == L) {
      float cum = before + inc - ls;
      int pick = -1, last = s0;
      bool tie = !hit;
      for (int x = s0; x < s1; ++x) {
        const float wv = fast_exp2(__ldcg(row + x) * l2s - M);
        if (wv > 0.f) last = x;
        if (pick < 0 && hit && cum + wv > target) {
          pick = x;
          tie = fabsf(target - cum) < kTieBand * S || fabsf(target - (cum + wv)) < kTieBand * S;
        }
        cum += wv;
      }
      if (pick < 0) {   // rounding: the last entry of positive weight, on the boundary
        pick = last;
        tie = true;
      }
      ts.leaf[4] = pick | (tie ? (1 << 31) : 0);
    }
  }
  __syncthreads();
  result = ts.leaf[4];
  return result;
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


// A node's tree context is read in one round trip: the parents and tokens of
// nodes t-127 .. t+127 (a request holds at most 128 nodes) and the offsets.
// tree_loads() issues this thread's share of those loads into registers, so
// a kernel can issue them before its bulk row loads and let load_tree()
// consume them afterwards.
struct TreeLoads {
  int par, tok, o0, o1;
};

__device__ __forceinline__ TreeLoads tree_loads(const VerifyArgs &a, int t) {
  const int tid = threadIdx.x;
  TreeLoads r{-2, 0, 0, 0};
  if (tid < kTreeWindow) {
    const int x = t - (SPEC_MAX_TREE_NODES - 1) + tid;
    if (x >= 0 && x < a.T) {
      r.par = __ldg(a.parents + x);
      r.tok = __ldg(a.tokens + x);
    }
  }
  if (tid < a.B) {
    r.o0 = __ldg(a.offsets + tid);
    r.o1 = __ldg(a.offsets + tid + 1);
  }
  return r;
}

// Phase A of load_tree, called by every thread of the CTA (blockDim >= 256)
// with its tree_loads(): stage the window and find node t's request.  One
// barrier.
static __device__ NodeCtx load_tree_a(const VerifyArgs &a, int t, TreeSmem &ts, const TreeLoads &ld) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  if (tid < kTreeWindow) {
    ts.wpar[tid] = ld.par;
    ts.wtok[tid] = ld.tok;
  }
  if (tid == 0) ts.timeout = 0;
  // The offsets must start at 0, never decrease and end at T; then exactly
  // one request owns t.
  int match = -1;
  bool bad = false;
  for (int i = tid; i < a.B; i += static_cast<int>(blockDim.x)) {
    const int o0 = i == tid ? ld.o0 : __ldg(a.offsets + i);
    const int o1 = i == tid ? ld.o1 : __ldg(a.offsets + i + 1);
    bad |= (o1 < o0) || (i == 0 && o0 != 0) || (i == a.B - 1 && o1 != a.T);
    if (o0 <= t && t < o1) {
      match = i;
      ts.meta[2] = o0;
      ts.meta[3] = o1 - o0;
    }
  }
  match = __reduce_max_sync(0xffffffffu, match);
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    ts.wmatch[w] = match;
    ts.wbad[w] = bad ? 1 : 0;
  }
  __syncthreads();
  match = __reduce_max_sync(0xffffffffu, lane < nwarps ? ts.wmatch[lane] : -1);
  bad = __any_sync(0xffffffffu, lane < nwarps && ts.wbad[lane] != 0);
  NodeCtx c;
  c.b = match;
  c.lo = c.n = c.k = 0;
  c.err = 0;
  c.count = !bad && match >= 0;
  if (!c.count) {
    c.err = SPEC_ERR_TREE_TOO_LARGE;
  } else {
    c.lo = ts.meta[2];
    c.n = ts.meta[3];
    if (c.n < 1 || c.n > SPEC_MAX_TREE_NODES) c.err = SPEC_ERR_TREE_TOO_LARGE;
  }
  c.u = t - c.lo;
  return c;
}

// Whether u has a child, from the staged window (nodes t+1 .. t+127 of the
// request whose parent is u); every warp computes it, no barrier.  Exact for
// a valid tree; load_tree_b() validates.
__device__ __forceinline__ bool has_children(const NodeCtx &c, int t, const TreeSmem &ts) {
  if (c.err) return false;
  const int lane = threadIdx.x & 31;
  bool hit = false;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int j = lane + 32 * s;   // node t + 1 + j, window slot 128 + j
    if (j < SPEC_MAX_TREE_NODES - 1 && t + 1 + j < c.lo + c.n) hit |= ts.wpar[SPEC_MAX_TREE_NODES + j] == c.u;
  }
  return __any_sync(0xffffffffu, hit);
}

// Phase B: one warp validates the request's parents and children's tokens
// and lists u's children in index order.  One barrier.
static __device__ NodeCtx load_tree_b(const VerifyArgs &a, int t, TreeSmem &ts, NodeCtx c) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (!c.err && w == 0) {
    bool bad_parent = false, bad_token = false;
    int k = 0;
#pragma unroll
    for (int s = 0; s < SPEC_MAX_TREE_NODES / 32; ++s) {
      const int i = lane + 32 * s;
      bool is_child = false;
      if (i < c.n) {
        const int wi = c.lo + i - (t - (SPEC_MAX_TREE_NODES - 1));   // in [0, 254]
        const int p = ts.wpar[wi];
        const int x = ts.wtok[wi];
        ts.par[i] = p;
        ts.tok[i] = x;
        bad_parent |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
        is_child = i > c.u && p == c.u;
        bad_token |= is_child && (x < 0 || x >= a.V);
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, is_child);
      if (is_child) ts.child[k + __popc(bal & ((1u << lane) - 1u))] = i;
      k += __popc(bal);
    }
    bad_parent = __any_sync(0xffffffffu, bad_parent);
    bad_token = __any_sync(0xffffffffu, bad_token);
    if (lane == 0) {
      ts.meta[0] = bad_parent ? SPEC_ERR_BAD_PARENT : (bad_token ? SPEC_ERR_TOKEN_RANGE : 0);
      ts.meta[1] = k;
    }
  }
  __syncthreads();  // child list complete
  if (!c.err) {
    c.err = ts.meta[0];
    c.k = ts.meta[1];
  }
  if (c.err) c.k = 0;
  return c;
}

// Both phases: find node t's request, stage its parents and tokens, validate
// them, and list u's children.  Errors are identical in every CTA of a group.
static __device__ NodeCtx load_tree(const VerifyArgs &a, int t, TreeSmem &ts, const TreeLoads &ld) {
  return load_tree_b(a, t, ts, load_tree_a(a, t, ts, ld));
}

// The request's parents and tokens from node t's staged window into ts.par /
// ts.tok, without validation (a node whose CTAs skip load_tree_b: the root,
// which validates, arrives with the error bit if the tree is malformed, and
// then no walk reads them).  Ends with a barrier.
static __device__ void stage_request(const NodeCtx &c, int t, TreeSmem &ts) {
  for (int i = threadIdx.x; i < c.n; i += blockDim.x) {
    const int wi = c.lo + i - (t - (SPEC_MAX_TREE_NODES - 1));   // in [0, 254]
    ts.par[i] = ts.wpar[wi];
    ts.tok[i] = ts.wtok[wi];
  }
  __syncthreads();
}

// The root's arrival when its walk is known to end at the root (every child
// of the root rejected, a valid tree, no wait of the CTA ran out, the path
// fits the output rows): it needs no other node's results, so the CTA that
// will draw the emitted token arrives before drawing it, and the atomic's
// round trip overlaps the draw.  Called by every thread of that CTA, after
// warp 0 stored path_fits_quiet() in ts.fits;
// `done` holds in warp 0, `prev` (the arrival word before) in thread 0.
struct RootArrival {
  bool done;
  uint32_t prev;
};

static __device__ RootArrival root_arrive_early(const VerifyArgs &a, const NodeCtx &c, TreeSmem &ts) {
  RootArrival r{false, 0u};
  const int tid = threadIdx.x;
  if (tid < 32) r.done = ts.fits != 0;   // path_fits_quiet, taken while the rows loaded
  if (tid == 0 && r.done) {
    // nothing this node wrote is read by another node: no ordering needed
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(r.prev)
                 : "l"(a.done + c.b), "r"(1u | kArriveRootDone)
                 : "memory");
  }
  return r;
}

// Called by every thread of the one CTA per node that publishes the node's
// results, once they are written (flags of its children, its fallback).
// `root_stop_token` >= 0 at the root when no child of the root was accepted:
// the walk ends there, so this CTA writes the request's outputs at once (the
// token, `root_stop_ties` near-ties) and arrives with the root-done bit,
// needing no other node's results.  Otherwise the node arrives with release
// semantics, and the request's last arrival (acquire) walks it, unless the
// root already wrote the outputs or a node's wait ran out.  The last arrival
// clears the request's counter for the next call (with valid offsets every
// node of the request arrives exactly once).
static __device__ void arrive_and_walk(const VerifyArgs &a, const NodeCtx &c, TreeSmem &ts,
                                       int root_stop_token, int root_stop_ties, bool timed_out,
                                       bool lazy_leaves = false,
                                       const RootArrival &early = RootArrival{false, 0u}) {
  const int tid = threadIdx.x;
  bool root_done = false;
  if (tid < 32 && early.done) {
    // the root arrived early (root_arrive_early): its outputs alone remain
    write_root_stop(a, c.b, root_stop_token, root_stop_ties);
    root_done = true;
  } else if (tid < 32 && c.count && !c.err && !timed_out && c.u == 0 && root_stop_token >= 0 &&
             path_fits(a, c.b, c.n, ts.par)) {
    write_root_stop(a, c.b, root_stop_token, root_stop_ties);
    root_done = true;
  }
  if (tid == 0) {
    int walk = 0;
    if (c.count) {
      // a node that found an error arrives with the error bit, so that no
      // walk (which trusts the validated tree) runs for the request
      const uint32_t add = 1u | ((timed_out || c.err) ? kArriveErr : 0u) |
                           (root_done ? kArriveRootDone : 0u);
      uint32_t prev;
      if (early.done) {
        prev = early.prev;
      } else if (root_done) {
        // nothing this node wrote is read by another node: no ordering needed
        asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;"
                     : "=r"(prev)
                     : "l"(a.done + c.b), "r"(add)
                     : "memory");
      } else {
        // release: this CTA's results (ordered before by the caller's
        // barrier); acquire: every earlier arrival's results
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                     : "=r"(prev)
                     : "l"(a.done + c.b), "r"(add)
                     : "memory");
      }
      if (static_cast<int>(prev & kArriveCount) == c.n - 1) {
        a.done[c.b] = 0u;
        const uint32_t all = prev + add;
        walk = (!c.err && !(all & kArriveErrMask) && !(all & kArriveRootDone)) ? 1 : 0;
      }
    }
    ts.walk = walk;
  }
  __syncthreads();
  // The walker's loads are ordered after thread 0's acquire by the barrier
  // and read L2 (ld.global.cg), where the other nodes' released results sit.
  if (!ts.walk) return;
  if (tid == 0) ts.leaf[0] = -1;
  __syncthreads();
  if (tid < 32) walk_request(a, c.b, c.lo, c.n, ts.par, ts.tok, lazy_leaves, ts);
  __syncthreads();
  const int leaf = ts.leaf[0];
  if (leaf < 0) return;
  // the walk accepted the path down to a leaf: the bonus token is its draw
  if (!in_bounds(c.lo + leaf, a.T, a.status, c.b)) return;   // CTA-uniform
  const float *row = a.target + static_cast<size_t>(c.lo + leaf) * a.V;
  const int r = cta_leaf_draw(row, a.V, a.inv_temp * 1.4426950408889634f,
                              spec_uniform(a.seed, leaf, c.b, 1), ts);
  if (tid == 0 && in_bounds(ts.leaf[1], a.W, a.status, c.b)) {
    a.out_tokens[static_cast<size_t>(c.b) * a.W + ts.leaf[1]] = r & 0x7fffffff;
    a.near_ties[c.b] = ts.leaf[2] + ((r >> 31) & 1);
  }
}

// Host entry of spec_tree_verify / spec_tree_verify_top_p (verify.cu): checks
// every argument on the host, then, when clear_workspace is set, zero-fills
// the workspace's used bytes on `stream`, then launches.  Nothing is enqueued
// when a check fails.
int verify_entry(const float *target_logits, const float *draft_logits, const int32_t *tokens,
                 const int32_t *parents, const int32_t *tree_offsets, int B, int T, int V,
                 float temperature, float top_p, uint64_t seed, int32_t *accept_len,
                 int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                 void *workspace, size_t workspace_bytes, int32_t *status, void *stream,
                 bool clear_workspace, uint64_t wait_ns = kWaitLimitNs, int drop_request = -1);

// greedy per-node kernel (verify_node.cu)
int launch_verify_greedy(const VerifyArgs &args, cudaStream_t stream);

// stochastic kernel with the rows in registers (verify_reg.cu): CTAs of
// kRegChunk vocabulary entries, `cs` = ceil(V / kRegChunk) <= kMaxCS per node
constexpr int kRegChunk = 16384;
int launch_verify_reg(const VerifyArgs &args, int cs, bool top_p, cudaStream_t stream);

}  // namespace spec
