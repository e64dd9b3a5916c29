// Steps V1-V4 and R: verification of a speculated token tree.
//
// Sources: speculative-decoding explainer (intelliparadigm.com) §2.2
// 三阶段工作流程详解 — stage 2: accept probability alpha = min(1, p/q); stage 3:
// check left to right, stop at the first rejection and replace it with a new
// target prediction (output distribution equal to the target's).  SpecInfer
// developer article §2.1: the accept stage keeps the longest verified prefix.
//
// Parallel structure.  Which node the walk stops at is only known at the end,
// but everything a node contributes is fixed beforehand: its children are
// always tested in index order against the residual left by their earlier
// siblings, so the accept decision of every child and the token emitted when
// the walk stops at a node can all be computed at once, one node per
// thread-block cluster.  The last cluster of a request to finish then walks
// the tree in one warp.
//
// Residual chain in closed form.  With r_0 = p and r_j = norm(max(0,
// r_{j-1} - q)), induction gives r_j = max(0, p - c_j q) / W(c_j) with
// W(c) = sum_v max(0, p(v) - c q(v)), c_0 = 0, W(c_0) = 1 and
// c_j = c_{j-1} + W(c_{j-1}).  So each rejection costs one cluster-wide
// reduction over the vocabulary held in shared memory, and the accept test of
// the j-th child is alpha_j = min(1, max(0, p(x) - c_{j-1} q(x)) /
// (W(c_{j-1}) q(x))).  A residual that sums to zero (r == q up to rounding)
// leaves r unchanged, i.e. keeps c.
#include <cooperative_groups.h>

#include "common.cuh"

namespace spec {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kMaxCS = 8;          // CTAs per cluster (portable limit)
constexpr int kMaxChunk = 27648;   // floats per CTA per row (2 rows fit in 216 KB)
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
  int32_t *flags;      // [T] written by the parent's cluster: accept / tie bits
  int32_t *fallback;   // [T] token emitted on stopping at the node | tie << 31
  uint32_t *done;      // [B] arrival counters, then one global counter at [B]
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
__device__ void walk_request(const VerifyArgs &a, int b, int lo, int n, const int *spar,
                             const int *stok) {
  const int lane = threadIdx.x & 31;
  if (*reinterpret_cast<volatile int32_t *>(a.status + b) != 0) return;
  int par[4], flg[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int i = lane + 32 * s;
    par[s] = i < n ? spar[i] : -2;
    flg[s] = i < n ? __ldcg(a.flags + lo + i) : 0;
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
      const int fb = __ldcg(a.fallback + lo + cur);
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

// Per-CTA scratch for one reduction round, double buffered by round parity
// so a round never waits for the previous round's readers.
struct RoundScratch {
  float w[2][kVWarps][2];
  int wi[2][kVWarps];
};

// Cluster all-gather slots: every CTA pushes its partials into slot [rank]
// of every peer with remote stores, so after one cluster barrier all values
// are read from local shared memory.  Double buffered by round parity.
struct Gather {
  float v[2][kMaxCS][4];
};

__device__ __forceinline__ void gather_push(Gather &gx, int parity, int rank, int CS, float4 val) {
  // threads 0..CS-1 each push to one peer
  const int r = threadIdx.x;
  if (r < CS) st_peer_f32x4(peer_addr(&gx.v[parity][rank][0], r), val);
}

// Sum `x` over the CTA and then over the cluster.  Returns the cluster total
// (identical in every CTA: partials are added in rank order) and, in `parts`,
// the per-CTA totals.  One __syncthreads and one cluster barrier.
__device__ float cluster_round_sum(float x, RoundScratch &rs, Gather &gx, int parity, int rank,
                                   int CS, float *parts) {
  x = warp_sum(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) rs.w[parity][w][0] = x;
  __syncthreads();
  if (threadIdx.x < CS) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kVWarps; ++i) t += rs.w[parity][i][0];
    gather_push(gx, parity, rank, CS, make_float4(t, 0.f, 0.f, 0.f));
  }
  cluster_sync_all();
  float tot = 0.f;
  for (int r = 0; r < CS; ++r) {
    const float v = gx.v[parity][r][0];
    if (parts) parts[r] = v;
    tot += v;
  }
  return tot;
}

__global__ void __launch_bounds__(kVThreads)
tree_verify_kernel(const VerifyArgs a) {
  extern __shared__ __align__(128) float vsm[];  // [chunk] target side, [chunk] draft side
  __shared__ RoundScratch rs;
  __shared__ __align__(16) Gather gx;           // cluster all-gather, double buffered
  __shared__ int spar[SPEC_MAX_TREE_NODES];
  __shared__ int stok[SPEC_MAX_TREE_NODES];
  __shared__ int child_id[SPEC_MAX_TREE_NODES];
  __shared__ float childP[SPEC_MAX_TREE_NODES], childQ[SPEC_MAX_TREE_NODES];
  __shared__ float childU[SPEC_MAX_TREE_NODES];
  __shared__ int warp_cnt[4];
  __shared__ int s_meta[4];                     // error, request, n_children
  __shared__ float s_ufb;
  __shared__ int s_walk, s_pick;
  __shared__ float s_cb[2];
  __shared__ __align__(8) uint64_t bars[2];

  const int CS = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_rank());
  const int t = blockIdx.x / CS;
  const int tid = threadIdx.x, w_id = tid >> 5, lane = tid & 31;
  float *lrow = vsm;
  float *drow = vsm + a.chunk;
  const int v0 = rank * a.chunk;
  const int len = max(0, min(a.V, v0 + a.chunk) - v0);
  const bool greedy = !(a.temp > 0.f);
  // 1-D bulk copies need 16-byte aligned rows and a length multiple of 16 B.
  const bool bulk = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0) &&
                    (greedy || (reinterpret_cast<uintptr_t>(a.draft) & 15) == 0);
  const float *trow_g = a.target + static_cast<size_t>(t) * a.V;
  const float *drow_g = greedy ? nullptr : a.draft + static_cast<size_t>(t) * a.V;

  // ---- V1 (start): the target row slice streams in while the tree is read
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
    s_meta[0] = 0;
    s_meta[1] = -1;
    if (bulk && len > 0) {
      mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(len) * 4u);
      bulk_copy_g2s(lrow, trow_g + v0, static_cast<uint32_t>(len) * 4u, &bars[0]);
    }
  }
  // ---- locate the node's request (identical in every CTA of the cluster)
  if (a.B < kVThreads) {
    if (tid < a.B) {
      const int o0 = __ldg(a.offsets + tid), o1 = __ldg(a.offsets + tid + 1);
      if (o0 <= t && t < o1) atomicMax(&s_meta[1], tid);
    }
  } else if (tid == 0) {
    s_meta[1] = find_request(a.offsets, a.B, t);
  }
  __syncthreads();
  const int b = s_meta[1];
  int lo = 0, n = 0, err = 0;
  if (b < 0) {
    err = SPEC_ERR_TREE_TOO_LARGE;
  } else {
    lo = __ldg(a.offsets + b);
    n = __ldg(a.offsets + b + 1) - lo;
    if (lo < 0 || lo + n > a.T || n < 1 || n > SPEC_MAX_TREE_NODES) err = SPEC_ERR_TREE_TOO_LARGE;
  }
  const int u = t - lo;
  // ---- the request's tree: parents, tokens, and u's children in index order
  bool is_child = false;
  uint32_t child_bal = 0;
  if (!err && tid < SPEC_MAX_TREE_NODES) {
    int p = -2, x = 0;
    if (tid < n) {
      p = __ldg(a.parents + lo + tid);
      x = __ldg(a.tokens + lo + tid);
      spar[tid] = p;
      stok[tid] = x;
      const bool ok = (tid == 0) ? (p == -1) : (p >= 0 && p < tid);
      if (!ok) atomicCAS(&s_meta[0], 0, SPEC_ERR_BAD_PARENT);
      is_child = (tid > u && p == u);
      if (is_child && (x < 0 || x >= a.V)) atomicCAS(&s_meta[0], 0, SPEC_ERR_TOKEN_RANGE);
    }
    child_bal = __ballot_sync(0xffffffffu, is_child);
    if (lane == 0) warp_cnt[w_id] = __popc(child_bal);
  }
  __syncthreads();
  if (!err) err = s_meta[0];
  int k = 0;
  if (!err) {
    int before = 0;
    for (int i = 0; i < SPEC_MAX_TREE_NODES / 32; ++i) {
      if (i < w_id) before += warp_cnt[i];
      k += warp_cnt[i];
    }
    if (is_child) child_id[before + __popc(child_bal & ((1u << lane) - 1u))] = tid;
  }
  const bool need_draft = !err && !greedy && k > 0;
  if (tid == 0 && bulk && need_draft && len > 0) {
    mbar_arrive_expect_tx(&bars[1], static_cast<uint32_t>(len) * 4u);
    bulk_copy_g2s(drow, drow_g + v0, static_cast<uint32_t>(len) * 4u, &bars[1]);
  }
  __syncthreads();  // child_id complete
  // the draws and the children's logits at their tokens, in parallel
  if (!err && !greedy) {
    if (tid < k) {
      const int c = child_id[tid];
      const int x = stok[c];
      childP[tid] = __ldg(trow_g + x);
      childQ[tid] = __ldg(drow_g + x);
      childU[tid] = spec_uniform(a.seed, c, b, 0);
    } else if (tid == kVThreads - 1) {
      s_ufb = spec_uniform(a.seed, u, b, 1);
    }
  }
  // ---- wait for the slices (a copy issued for a node is always waited for)
  bool timed_out = false;
  if (bulk && len > 0) {
    if (!mbar_wait(&bars[0], 0)) timed_out = true;
    if (need_draft && !mbar_wait(&bars[1], 0)) timed_out = true;
  } else if (!err) {
    for (int i = tid; i < len; i += kVThreads) {
      lrow[i] = __ldcs(trow_g + v0 + i);
      if (need_draft) drow[i] = __ldcs(drow_g + v0 + i);
    }
  }
  if (timed_out && tid == 0) report(a.status, b, SPEC_ERR_TIMEOUT);
  __syncthreads();

  if (!err) {
    int parity = 0;
    if (greedy) {
      // ---- argmax of the raw target logits, lowest index on ties
      ArgMax am{-INFINITY, 0x7fffffff};
      for (int i = tid; i < len; i += kVThreads) am = better(am, ArgMax{lrow[i], v0 + i});
      am = warp_argmax(am);
      if (lane == 0) {
        rs.w[0][w_id][0] = am.v;
        rs.wi[0][w_id] = am.i;
      }
      __syncthreads();
      if (tid < CS) {
        ArgMax r{rs.w[0][0][0], rs.wi[0][0]};
        for (int i = 1; i < kVWarps; ++i) r = better(r, ArgMax{rs.w[0][i][0], rs.wi[0][i]});
        gather_push(gx, 0, rank, CS, make_float4(r.v, __int_as_float(r.i), 0.f, 0.f));
      }
      cluster_sync_all();
      if (rank == 0 && tid == 0) {
        ArgMax g{-INFINITY, 0x7fffffff};
        for (int r = 0; r < CS; ++r) g = better(g, ArgMax{gx.v[0][r][0], __float_as_int(gx.v[0][r][1])});
        a.fallback[t] = g.i;
        for (int j = 0; j < k; ++j) {
          const int c = child_id[j];
          a.flags[lo + c] = (stok[c] == g.i) ? kFlagAccept : 0;
        }
      }
    } else {
      const float T_ = a.temp, iT = a.inv_temp;
      // ---- V1: per-thread max and sum of exp((x - m)/T) over the thread's
      //      elements, combined over the CTA and the cluster in one round
      float ml = -INFINITY, md = -INFINITY;
      for (int i = tid; i < len; i += kVThreads) {
        ml = fmaxf(ml, lrow[i]);
        if (need_draft) md = fmaxf(md, drow[i]);
      }
      float sl = 0.f, sd = 0.f;
      for (int i = tid; i < len; i += kVThreads) {
        const float el = expf((lrow[i] - ml) * iT);
        lrow[i] = el;
        sl += el;
        if (need_draft) {
          const float ed = expf((drow[i] - md) * iT);
          drow[i] = ed;
          sd += ed;
        }
      }
      // warp combine of (m, s) pairs
      float wml = warp_max(ml), wmd = warp_max(md);
      float wsl = warp_sum(sl > 0.f ? sl * expf((ml - wml) * iT) : 0.f);
      float wsd = warp_sum(sd > 0.f ? sd * expf((md - wmd) * iT) : 0.f);
      __shared__ float s_pair[kVWarps][4];
      if (lane == 0) {
        s_pair[w_id][0] = wml;
        s_pair[w_id][1] = wsl;
        s_pair[w_id][2] = wmd;
        s_pair[w_id][3] = wsd;
      }
      __syncthreads();
      if (tid < CS) {
        float cm = -INFINITY, cmd = -INFINITY;
        for (int i = 0; i < kVWarps; ++i) {
          cm = fmaxf(cm, s_pair[i][0]);
          cmd = fmaxf(cmd, s_pair[i][2]);
        }
        float cs = 0.f, csd = 0.f;
        for (int i = 0; i < kVWarps; ++i) {
          if (s_pair[i][1] > 0.f) cs += s_pair[i][1] * expf((s_pair[i][0] - cm) * iT);
          if (s_pair[i][3] > 0.f) csd += s_pair[i][3] * expf((s_pair[i][2] - cmd) * iT);
        }
        gather_push(gx, parity, rank, CS, make_float4(cm, cs, cmd, csd));
      }
      cluster_sync_all();
      float Ml = -INFINITY, Md = -INFINITY;
      float4 part[kMaxCS];
      for (int r = 0; r < CS; ++r) {
        part[r] = *reinterpret_cast<const float4 *>(&gx.v[parity][r][0]);
        Ml = fmaxf(Ml, part[r].x);
        Md = fmaxf(Md, part[r].z);
      }
      float Sp = 0.f, Sq = 0.f;
      float kept[kMaxCS];
      for (int r = 0; r < CS; ++r) {
        kept[r] = part[r].y > 0.f ? part[r].y * expf((part[r].x - Ml) * iT) : 0.f;
        Sp += kept[r];
        if (need_draft && part[r].w > 0.f) Sq += part[r].w * expf((part[r].z - Md) * iT);
      }
      for (int r = 0; r < CS; ++r) kept[r] /= Sp;  // chunk sums of p
      parity ^= 1;
      // p(v), q(v) for this thread's elements
      const float scale_l = ml == -INFINITY ? 0.f : expf((ml - Ml) * iT) / Sp;
      const float scale_d = (need_draft && md != -INFINITY) ? expf((md - Md) * iT) / Sq : 0.f;
      for (int i = tid; i < len; i += kVThreads) {
        lrow[i] *= scale_l;
        if (need_draft) drow[i] *= scale_d;
      }

      // ---- V2: the children's accept tests, one reduction per rejection
      float c_prev = 0.f, W_prev = 1.f;
      for (int j = 0; j < k; ++j) {
        const int c = child_id[j];
        const float P = precise_prob(childP[j], Ml, T_, iT, Sp);
        const float Q = precise_prob(childQ[j], Md, T_, iT, Sq);
        const float alpha = Q > 0.f ? fminf(1.f, fmaxf(0.f, fmaf(-c_prev, Q, P)) / (W_prev * Q)) : 1.f;
        if (rank == 0 && tid == 0) {
          const float uu = childU[j];
          int f = (uu < alpha) ? kFlagAccept : 0;
          if (fabsf(uu - alpha) < kTieBand) f |= kFlagTie;
          a.flags[lo + c] = f;
        }
        const float c_new = c_prev + W_prev;
        float w = 0.f;
        for (int i = tid; i < len; i += kVThreads) w += fmaxf(0.f, fmaf(-c_new, drow[i], lrow[i]));
        float chunks[kMaxCS];
        const float Wn = cluster_round_sum(w, rs, gx, parity, rank, CS, chunks);
        parity ^= 1;
        if (Wn > 0.f) {  // otherwise the residual is all zero: keep r
          c_prev = c_new;
          W_prev = Wn;
          for (int r = 0; r < CS; ++r) kept[r] = chunks[r];
        }
      }

      // ---- V3: the token emitted when the walk stops here, drawn by
      //      inverse CDF from r ∝ max(0, p - c q) (c = 0: r = p)
      float total = 0.f;
      for (int r = 0; r < CS; ++r) total += kept[r];
      const float target = s_ufb * total;
      int owner = -1;
      float prefix = 0.f;
      {
        float run = 0.f;
        for (int r = 0; r < CS; ++r) {
          if (run + kept[r] > target) { owner = r; prefix = run; break; }
          run += kept[r];
        }
        if (owner < 0) {  // rounding kept the running sum below the target
          run = 0.f;
          for (int r = 0; r < CS; ++r) {
            if (kept[r] > 0.f) { owner = r; prefix = run; }
            run += kept[r];
          }
        }
      }
      if (rank == owner) {
        // Warp-contiguous segments; warp partial sums, then the owning warp
        // scans its segment 32 elements at a time.
        const int seg = (len + kVWarps - 1) / kVWarps;
        const int s0 = min(len, w_id * seg), s1 = min(len, s0 + seg);
        float ws = 0.f;
        for (int i = s0 + lane; i < s1; i += 32)
          ws += c_prev != 0.f ? fmaxf(0.f, fmaf(-c_prev, drow[i], lrow[i])) : lrow[i];
        ws = warp_sum(ws);
        if (lane == 0) rs.w[parity][w_id][1] = ws;
        if (tid == 0) s_pick = -1;
        __syncthreads();
        float before = prefix;
        int pick_w = -1;
        {
          float run = prefix;
          for (int i = 0; i < kVWarps; ++i) {
            if (run + rs.w[parity][i][1] > target) { pick_w = i; before = run; break; }
            run += rs.w[parity][i][1];
          }
        }
        if (pick_w == w_id) {
          float run = before;
          for (int base = s0; base < s1; base += 32) {
            const int i = base + lane;
            float wv = 0.f;
            if (i < s1) wv = c_prev != 0.f ? fmaxf(0.f, fmaf(-c_prev, drow[i], lrow[i])) : lrow[i];
            float inc = wv;  // inclusive warp scan
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, inc, o);
              if (lane >= o) inc += y;
            }
            const float cum = run + inc;
            const uint32_t hit = __ballot_sync(0xffffffffu, i < s1 && cum > target);
            if (hit) {
              if (lane == __ffs(hit) - 1) {
                s_pick = v0 + i;
                s_cb[0] = cum - wv;
                s_cb[1] = cum;
              }
              break;
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
          }
        }
        __syncthreads();
        if (tid == 0) {
          int pick = s_pick;
          float cb0, cb1;
          if (pick >= 0) {
            cb0 = s_cb[0];
            cb1 = s_cb[1];
          } else {  // not reached in this slice: last positive weight of the slice
            for (int i = len - 1; i >= 0; --i) {
              const float wv = c_prev != 0.f ? fmaxf(0.f, fmaf(-c_prev, drow[i], lrow[i])) : lrow[i];
              if (wv > 0.f) { pick = v0 + i; break; }
            }
            if (pick < 0) pick = v0;
            cb0 = cb1 = target;  // the draw sits on the boundary
          }
          const bool tie = fabsf(target - cb0) < kTieBand * total || fabsf(target - cb1) < kTieBand * total;
          a.fallback[t] = pick | (tie ? (1 << 31) : 0);
          __threadfence();
        }
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its exchange slots
  } else if (rank == 0 && tid == 0 && b >= 0) {
    report(a.status, b, err);
  }

  // ---- arrival: the last cluster of a request walks it; the last cluster
  //      of the grid clears every counter for the next call
  if (rank == 0) {
    if (tid == 0) {
      __threadfence();
      int walk = 0;
      if (b >= 0) {
        const uint32_t prev = atomicAdd(a.done + b, 1u);
        walk = (!err && static_cast<int>(prev) == n - 1) ? 1 : 0;
      }
      s_walk = walk;
    }
    __syncthreads();
    if (s_walk) {
      __threadfence();
      if (tid < 32) walk_request(a, b, lo, n, spar, stok);
    }
    if (tid == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(a.done + a.B, 1u);
      if (prev == gridDim.x / CS - 1) {
        for (int i = 0; i <= a.B; ++i) a.done[i] = 0u;
      }
    }
  }
}

}  // namespace spec

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}

extern "C" size_t spec_tree_verify_workspace_size(int B, int T, int V) {
  (void)V;
  if (B < 1 || T < 1) return 0;
  return align256(sizeof(uint32_t) * (B + 1)) + align256(sizeof(int32_t) * T) * 2;
}

extern "C" int spec_tree_verify(const float *target_logits, const float *draft_logits,
                                const int32_t *tokens, const int32_t *parents,
                                const int32_t *tree_offsets, int B, int T, int V,
                                float temperature, uint64_t seed, int32_t *accept_len,
                                int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties,
                                int max_depth_plus1, void *workspace, size_t workspace_bytes,
                                int32_t *status, void *stream) {
  using namespace spec;
  if (!target_logits || !tokens || !parents || !tree_offsets || !accept_len || !path_nodes ||
      !out_tokens || !near_ties || !status)
    return SPEC_ERR_NULL;
  if (B < 1 || T < 1 || T > B * SPEC_MAX_TREE_NODES || V < 1 || max_depth_plus1 < 1)
    return SPEC_ERR_SHAPE;
  if (!(temperature >= 0.f) || temperature > 1e4f) return SPEC_ERR_SHAPE;  // rejects NaN too
  const bool greedy = temperature == 0.f;
  if (!greedy && !draft_logits) return SPEC_ERR_NULL;
  const size_t need = spec_tree_verify_workspace_size(B, T, V);
  if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return SPEC_ERR_ALIGNMENT;

  int CS = (V + 4095) / 4096;
  if (CS > kMaxCS) CS = kMaxCS;
  if (CS < 1) CS = 1;
  int chunk = (V + CS - 1) / CS;
  chunk = (chunk + 3) & ~3;
  if (chunk > kMaxChunk) return SPEC_ERR_SHAPE;

  VerifyArgs args;
  args.target = target_logits;
  args.draft = draft_logits;
  args.tokens = tokens;
  args.parents = parents;
  args.offsets = tree_offsets;
  args.B = B;
  args.T = T;
  args.V = V;
  args.chunk = chunk;
  args.W = max_depth_plus1;
  args.temp = temperature;
  args.inv_temp = greedy ? 0.f : 1.0f / temperature;
  args.seed = seed;
  args.accept_len = accept_len;
  args.path_nodes = path_nodes;
  args.out_tokens = out_tokens;
  args.near_ties = near_ties;
  args.status = status;
  char *ws = static_cast<char *>(workspace);
  args.done = reinterpret_cast<uint32_t *>(ws);
  ws += align256(sizeof(uint32_t) * (B + 1));
  args.flags = reinterpret_cast<int32_t *>(ws);
  ws += align256(sizeof(int32_t) * T);
  args.fallback = reinterpret_cast<int32_t *>(ws);

  const size_t smem = sizeof(float) * 2 * static_cast<size_t>(chunk);
  static int configured_smem = -1;
  if (configured_smem < static_cast<int>(smem)) {
    if (cudaFuncSetAttribute(tree_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SPEC_ERR_CUDA;
    configured_smem = static_cast<int>(smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T) * CS, 1, 1);
  cfg.blockDim = dim3(kVThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tree_verify_kernel, args) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}
