// Steps V1-V4 and R: verification of a speculated token tree.  Greedy
// verification runs the per-node kernel of verify_node.cu; stochastic
// verification runs one thread-block cluster per node, with the node's rows
// in registers (verify_reg.cu) up to 131072 vocabulary entries, and for
// larger vocabularies split across the cluster's shared memory (the kernel
// below, up to 27648 entries per CTA).
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
// the walk stops at a node can all be computed at once, one node per CTA
// group.  A node's chain stops at its first accepted child (the walk never
// tests later children, nor draws at a node it leaves), so most nodes need
// no reduction round and no draw.  The last group of a request to finish
// then walks the tree in one warp.
//
// Residual chain in closed form.  With r_0 = p and r_j = norm(max(0,
// r_{j-1} - q)), induction gives r_j = max(0, p - c_j q) / W(c_j) with
// W(c) = sum_v max(0, p(v) - c q(v)), c_0 = 0, W(c_0) = 1 and
// c_j = c_{j-1} + W(c_{j-1}).  So each rejection costs one reduction over the
// vocabulary held on chip, and the accept test of the j-th child is
// alpha_j = min(1, max(0, p(x) - c_{j-1} q(x)) / (W(c_{j-1}) q(x))).  A
// residual that sums to zero (r == q up to rounding) leaves r unchanged, i.e.
// keeps c.
#include "verify_common.cuh"

namespace spec {

// Exchange slots of a node's CTA group.  Every warp pushes its partial sum
// into slot [rank][warp] of every CTA of the group with st.async, and the
// round's mbarrier in each CTA completes once all CS x 32 partials (in the
// statistics round also the slice maxima and the children's logits) have
// landed: no CTA-wide or cluster-wide barrier per round.  Every warp then
// adds the partials in the same order, so all threads of the group hold
// bit-identical totals.
struct Exchange {
  float2 statm[kMaxCS];                // per slice: max target logit, max draft logit
  float2 stat[kMaxCS][kVWarps];        // per warp: sums of 2^((x - max) * l2s), target and draft
  float part[2][kMaxCS][kVWarps];      // reduction rounds, by round parity
  float2 child[SPEC_MAX_TREE_NODES];   // the children's raw logits (target, draft)
};

__global__ void __launch_bounds__(kVThreads)
tree_verify_cluster_kernel(const VerifyArgs a) {
  extern __shared__ __align__(128) float vsm[];  // [chunk] target side, [chunk] draft side
  __shared__ __align__(16) Exchange ex;
  __shared__ TreeSmem ts;
  __shared__ float s_red[2][kVWarps];
  __shared__ float s_kept[kMaxCS];    // per slice: its share of p
  __shared__ float s_sc[2];
  __shared__ __align__(8) uint64_t bars[2];   // the slice copies
  __shared__ __align__(8) uint64_t xbar[3];   // exchange: statistics round, rounds by parity

  const int CS = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_rank());
  const int t = blockIdx.x / CS;
  const int tid = threadIdx.x, w_id = tid >> 5, lane = tid & 31;
  float *lrow = vsm;
  float *drow = vsm + a.chunk;
  const int v0 = rank * a.chunk;
  const int len = max(0, min(a.V, v0 + a.chunk) - v0);
  // Every pass gives warp w the contiguous range [e0, e1) of the slice (lanes
  // strided), so a pass's per-warp sums are also the first level of the
  // inverse-CDF search.
  const int seg = (((len + kVWarps - 1) / kVWarps) + 31) & ~31;
  const int e0 = min(len, w_id * seg), e1 = min(len, e0 + seg);
  // 1-D bulk copies need 16-byte aligned rows and a length multiple of 16 B.
  const bool bulk = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0) &&
                    ((reinterpret_cast<uintptr_t>(a.draft) & 15) == 0) && len > 0;
  const float *trow_g = a.target + static_cast<size_t>(t) * a.V;
  const float *drow_g = a.draft + static_cast<size_t>(t) * a.V;

  pdl_trigger();
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    for (int i = 0; i < 3; ++i) mbar_init(&xbar[i], 1);
    fence_barrier_init();
  }
  pdl_wait();
  const TreeLoads tl = tree_loads(a, t);   // issued ahead of the row copies
  // ---- V1 (start): the target row slice streams in while the tree is read
  if (tid == 0) {
    if (bulk) {
      mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(len) * 4u);
      bulk_copy_g2s(lrow, trow_g + v0, static_cast<uint32_t>(len) * 4u, &bars[0]);
    }
  }
  // waited for before the first remote store (the barriers are initialised)
  if (CS > 1) cluster_arrive_relaxed();
  const NodeCtx c = load_tree(a, t, ts, tl);
  const int k = c.k;
  const bool need_draft = !c.err && k > 0;   // leaves never read their draft row
  if (tid == 0 && bulk && need_draft) {
    mbar_arrive_expect_tx(&bars[1], static_cast<uint32_t>(len) * 4u);
    bulk_copy_g2s(drow, drow_g + v0, static_cast<uint32_t>(len) * 4u, &bars[1]);
  }
  if (!c.err) {
    // step R: the children's accept-test uniforms and the fallback draw's
    if (tid < k) ts.cU[tid] = spec_uniform(a.seed, ts.child[tid], c.b, 0);
    else if (tid == kVThreads - 1) ts.ufb = spec_uniform(a.seed, c.u, c.b, 1);
    if (tid == 0)
      mbar_arrive_expect_tx(&xbar[0], static_cast<uint32_t>(CS * (8 + kVWarps * 8) + 8 * k));
  }
  // ---- wait for the slices (a copy issued for a node is always waited for)
  bool ok = true;
  if (bulk) {
    if (!mbar_wait(&bars[0], 0)) ok = false;
    if (need_draft && !mbar_wait(&bars[1], 0)) ok = false;
  }
  if (CS > 1) cluster_wait();  // every CTA of the group is running
  if (!bulk && !c.err) {
    for (int i = tid; i < len; i += kVThreads) {
      lrow[i] = __ldcs(trow_g + v0 + i);
      if (need_draft) drow[i] = __ldcs(drow_g + v0 + i);
    }
  }
  // The children's raw logits, from the CTA whose slice holds them, to every
  // CTA of the group (read before the slices are overwritten below).
  if (need_draft && tid < k) {
    const int x = ts.tok[ts.child[tid]];
    if (x >= v0 && x < v0 + len) {
      const float pl = bulk ? lrow[x - v0] : __ldg(trow_g + x);
      const float ql = bulk ? drow[x - v0] : __ldg(drow_g + x);
      for (int r = 0; r < CS; ++r)
        st_async_v2_f32(peer_addr(&ex.child[tid], r), pl, ql, peer_addr(&xbar[0], r));
    }
  }
  if (!bulk) __syncthreads();  // the plainly loaded slices are complete

  int stop = k;        // first accepted child, k when every child is rejected
  int my_flag = 0;     // thread j < k: the flag of child j
  int p_ok = -1;       // parity of the last reduction round that moved the residual
  float c_prev = 0.f, sc_l = 0.f, sc_d = 0.f;
  if (!c.err) {
    const float T_ = a.temp, iT = a.inv_temp;
    const float l2s = iT * 1.4426950408889634f;  // exp(x / T) = 2^(x * l2s)
    // ---- V1: the slice's maxima, then its exponentials in place (one scale
    //      per slice: p(v) = sc_l * lrow[v], q(v) = sc_d * drow[v])
    float ml = -INFINITY, md = -INFINITY;
    for (int i = e0 + lane; i < e1; i += 32) {
      ml = fmaxf(ml, lrow[i]);
      if (need_draft) md = fmaxf(md, drow[i]);
    }
    ml = warp_max(ml);
    md = warp_max(md);
    if (lane == 0) {
      s_red[0][w_id] = ml;
      s_red[1][w_id] = md;
    }
    __syncthreads();
    ml = warp_max(s_red[0][lane]);
    md = warp_max(s_red[1][lane]);
    float sl = 0.f, sd = 0.f;
    for (int i = e0 + lane; i < e1; i += 32) {
      const float el = fast_exp2((lrow[i] - ml) * l2s);
      lrow[i] = el;
      sl += el;
      if (need_draft) {
        const float ed = fast_exp2((drow[i] - md) * l2s);
        drow[i] = ed;
        sd += ed;
      }
    }
    sl = warp_sum(sl);
    sd = warp_sum(sd);
    if (lane < CS) {
      const uint32_t bar = peer_addr(&xbar[0], lane);
      st_async_v2_f32(peer_addr(&ex.stat[rank][w_id], lane), sl, sd, bar);
      if (w_id == 0) st_async_v2_f32(peer_addr(&ex.statm[rank], lane), ml, md, bar);
    }
    if (ok && !mbar_wait(&xbar[0], 0)) ok = false;
    if (w_id == 0) {
      // group maxima and sums, the slices' shares of p, the children's p and q
      float Ml = -INFINITY, Md = -INFINITY;
      for (int r = 0; r < CS; ++r) {
        Ml = fmaxf(Ml, ex.statm[r].x);
        Md = fmaxf(Md, ex.statm[r].y);
      }
      float Sp = 0.f, Sq = 0.f, mine = 0.f;
      for (int r = 0; r < CS; ++r) {
        const float2 v = ex.stat[r][lane];
        const float sp = warp_sum(v.x), sq = warp_sum(v.y);
        const float2 m = ex.statm[r];
        const float fp = sp > 0.f ? sp * fast_exp2((m.x - Ml) * l2s) : 0.f;
        Sp += fp;
        if (need_draft && sq > 0.f) Sq += sq * fast_exp2((m.y - Md) * l2s);
        if (lane == r) mine = fp;
      }
      if (lane < CS) s_kept[lane] = mine / Sp;
      for (int j = lane; j < k; j += 32) {
        ts.cP[j] = precise_prob(ex.child[j].x, Ml, T_, iT, Sp);
        ts.cQ[j] = precise_prob(ex.child[j].y, Md, T_, iT, Sq);
      }
      if (lane == 0) {
        s_sc[0] = ml == -INFINITY ? 0.f : fast_exp2((ml - Ml) * l2s) / Sp;
        s_sc[1] = (need_draft && md != -INFINITY) ? fast_exp2((md - Md) * l2s) / Sq : 0.f;
      }
    }
    __syncthreads();
    sc_l = s_sc[0];
    sc_d = s_sc[1];

    // ---- V2: the children's accept tests in index order.  The walk accepts
    //      the first accepted child, so the chain stops there: later children
    //      and this node's fallback draw can never be used.
    float W_prev = 1.f;
    bool frozen = false;   // a residual that summed to zero stays as it is
    int rounds = 0;
    for (int j = 0; j < k; ++j) {
      const float P = ts.cP[j];
      const float Q = ts.cQ[j];
      const float alpha = Q > 0.f ? fminf(1.f, fmaxf(0.f, fmaf(-c_prev, Q, P)) / (W_prev * Q)) : 1.f;
      const float uu = ts.cU[j];
      const bool accept = uu < alpha;
      if (tid == j) my_flag = (accept ? kFlagAccept : 0) | (fabsf(uu - alpha) < kTieBand ? kFlagTie : 0);
      if (accept) {
        stop = j;
        break;
      }
      if (frozen) continue;
      // After a wait ran out this thread takes part in no further exchange:
      // an arrival on a barrier whose previous phase never completed is not
      // allowed.  (Its request is reported and its walk not run.)
      if (!ok) {
        frozen = true;
        continue;
      }
      // rejected: r becomes max(0, p - c q) / W(c) with c = c_prev + W_prev
      const float c_new = c_prev + W_prev;
      const float cq = c_new * sc_d;
      float wsum = 0.f;
      for (int i = e0 + lane; i < e1; i += 32) wsum += fmaxf(0.f, fmaf(-cq, drow[i], sc_l * lrow[i]));
      wsum = warp_sum(wsum);
      const int p = rounds & 1;
      if (tid == 0) mbar_arrive_expect_tx(&xbar[1 + p], static_cast<uint32_t>(CS * kVWarps * 4));
      if (lane < CS)
        st_async_f32(peer_addr(&ex.part[p][rank][w_id], lane), wsum, peer_addr(&xbar[1 + p], lane));
      if (ok && !mbar_wait(&xbar[1 + p], (rounds >> 1) & 1)) ok = false;
      ++rounds;
      float Wn = 0.f;
      for (int r = 0; r < CS; ++r) Wn += warp_sum(ex.part[p][r][lane]);
      if (Wn > 0.f) {
        c_prev = c_new;
        W_prev = Wn;
        p_ok = p;
      } else {
        frozen = true;
      }
    }
  }
  // No CTA touches a peer's shared memory after this point: arrive now, wait
  // before exiting, so that no CTA leaves while a peer may still store to it.
  if (CS > 1) cluster_arrive_relaxed();
  if (!ok) {
    ts.timeout = 1;
    if (tid == 0) report(a.status, c.b, SPEC_ERR_TIMEOUT);
  }
  // A wait that ran out anywhere in the CTA: its threads may hold different
  // decisions, so the CTA takes one path from here on (no draw, no published
  // decision; rank 0 arrives with the error bit).
  const bool cta_timeout = __syncthreads_or(!ok);

  int writer = 0;  // the CTA of the group that publishes the node's results
  if (!c.err && !cta_timeout) {
    // ---- V3: when every child is rejected (or u is a leaf), the token
    //      emitted on stopping here: inverse CDF of r ∝ max(0, p - c q)
    if (stop == k) {
      float total = 0.f;
      for (int r = 0; r < CS; ++r)
        total += p_ok >= 0 ? warp_sum(ex.part[p_ok][r][lane]) : s_kept[r];
      const float target = ts.ufb * total;
      int owner = -1;
      float prefix = 0.f, run = 0.f;
      for (int r = 0; r < CS; ++r) {
        const float m = p_ok >= 0 ? warp_sum(ex.part[p_ok][r][lane]) : s_kept[r];
        if (owner < 0 && run + m > target) {
          owner = r;
          prefix = run;
        }
        run += m;
      }
      if (owner < 0) {  // rounding kept the running sum below the target
        run = 0.f;
        for (int r = 0; r < CS; ++r) {
          const float m = p_ok >= 0 ? warp_sum(ex.part[p_ok][r][lane]) : s_kept[r];
          if (m > 0.f) {
            owner = r;
            prefix = run;
          }
          run += m;
        }
        if (owner < 0) owner = 0;
      }
      writer = owner;
      if (rank == owner) {
        const float cq = c_prev * sc_d;
        auto weight = [&](int i) -> float {
          return c_prev != 0.f ? fmaxf(0.f, fmaf(-cq, drow[i], sc_l * lrow[i])) : sc_l * lrow[i];
        };
        auto scan = [&](float v) -> float {  // inclusive warp scan
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
          }
          return v;
        };
        // level 1: the slice's warp ranges, from the last pass's partials
        const float v1 = p_ok >= 0 ? ex.part[p_ok][rank][lane] : ex.stat[rank][lane].x * sc_l;
        const float inc1 = scan(v1);
        const uint32_t hit1 = __ballot_sync(0xffffffffu, prefix + inc1 > target);
        const int sw = hit1 ? __ffs(hit1) - 1 : -1;
        const float before1 = __shfl_sync(0xffffffffu, prefix + inc1 - v1, sw < 0 ? 0 : sw);
        // level 2: that range, one element per thread, 32-element groups
        const int g0 = sw < 0 ? 0 : min(len, sw * seg);
        const int g1 = sw < 0 ? 0 : min(len, g0 + seg);
        const int gi = g0 + tid;
        const float wv = gi < g1 ? weight(gi) : 0.f;
        const float gs = warp_sum(wv);
        if (lane == 0) s_red[1][w_id] = gs;
        __syncthreads();
        const float v2 = s_red[1][lane];
        const float inc2 = scan(v2);
        const uint32_t hit2 = __ballot_sync(0xffffffffu, before1 + inc2 > target);
        const int gw = (sw >= 0 && hit2) ? __ffs(hit2) - 1 : -1;
        if (gw >= 0 && w_id == gw) {
          // level 3: the group's elements
          const float before2 = __shfl_sync(0xffffffffu, before1 + inc2 - v2, gw);
          const float inc3 = scan(wv);
          const float cum = before2 + inc3;
          const uint32_t hit3 = __ballot_sync(0xffffffffu, gi < g1 && cum > target);
          int L;
          float cb0, cb1;
          if (hit3) {
            L = __ffs(hit3) - 1;
            cb0 = __shfl_sync(0xffffffffu, cum - wv, L);
            cb1 = __shfl_sync(0xffffffffu, cum, L);
          } else {  // rounding: the group's last positive weight, on the boundary
            const uint32_t pos = __ballot_sync(0xffffffffu, gi < g1 && wv > 0.f);
            L = pos ? 31 - __clz(pos) : 0;
            cb0 = cb1 = target;
          }
          if (lane == 0) {
            const bool tie = fabsf(target - cb0) < kTieBand * total || fabsf(target - cb1) < kTieBand * total;
            a.fallback[t] = (v0 + g0 + 32 * gw + L) | (tie ? (1 << 31) : 0);
            ts.stop_fb = (v0 + g0 + 32 * gw + L) | (tie ? (1 << 31) : 0);
          }
        } else if (gw < 0 && tid == 0) {
          // rounding: the slice's last positive weight, on the boundary
          int pick = -1;
          for (int i = len - 1; i >= 0; --i) {
            if (weight(i) > 0.f) {
              pick = v0 + i;
              break;
            }
          }
          if (pick < 0) pick = v0;
          a.fallback[t] = pick | (1 << 31);
          ts.stop_fb = pick | (1 << 31);
        }
      }
    }
    // every CTA computed the same decisions; the writer publishes them
    if (rank == writer && tid < k && in_bounds(c.lo + ts.child[tid], a.T, a.status, c.b))
      a.flags[c.lo + ts.child[tid]] = tid <= stop ? my_flag : 0;
  } else if (c.err && rank == 0 && tid == 0 && c.b >= 0) {
    report(a.status, c.b, c.err);
  }
  if (rank == writer) {
    // the node's flags and fallback are written; near-ties among the tested children
    const bool decided = !c.err && !cta_timeout;
    const int child_ties =
        __syncthreads_count(decided && tid < k && tid <= stop && (my_flag & kFlagTie) != 0);
    const int fb = ts.stop_fb;
    arrive_and_walk(a, c, ts, (decided && stop == k) ? (fb & 0x7fffffff) : -1,
                    child_ties + ((fb >> 31) & 1), cta_timeout);
  }
  if (CS > 1) cluster_wait();
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

namespace spec {
int verify_entry(const float *target_logits, const float *draft_logits, const int32_t *tokens,
                 const int32_t *parents, const int32_t *tree_offsets, int B, int T, int V,
                 float temperature, float top_p, uint64_t seed, int32_t *accept_len,
                 int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                 void *workspace, size_t workspace_bytes, int32_t *status, void *stream,
                 bool clear_workspace, uint64_t wait_ns, int drop_request) {
  if (!target_logits || !tokens || !parents || !tree_offsets || !accept_len || !path_nodes ||
      !out_tokens || !near_ties || !status)
    return SPEC_ERR_NULL;
  if (B < 1 || T < 1 || T > B * SPEC_MAX_TREE_NODES || V < 1 || max_depth_plus1 < 1)
    return SPEC_ERR_SHAPE;
  if (!(temperature >= 0.f) || temperature > 1e4f) return SPEC_ERR_SHAPE;  // rejects NaN too
  const bool greedy = temperature == 0.f;
  if (!greedy && !draft_logits) return SPEC_ERR_NULL;
  if (!(top_p > 0.f)) return SPEC_ERR_SHAPE;   // rejects NaN too
  const bool nucleus = !greedy && top_p < 1.f;   // the argmax is in every nucleus
  if (nucleus && V > kMaxCS * kRegChunk) return SPEC_ERR_SHAPE;
  const size_t need = spec_tree_verify_workspace_size(B, T, V);
  if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return SPEC_ERR_ALIGNMENT;

  int CS = (V + kChunkTarget - 1) / kChunkTarget;
  if (CS > kMaxCS) CS = kMaxCS;
  if (CS < 1) CS = 1;
  int chunk = (V + CS - 1) / CS;
  chunk = (chunk + 3) & ~3;
  if (!greedy && chunk > kMaxChunk) return SPEC_ERR_SHAPE;

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
  args.top_p = nucleus ? top_p : 1.f;
  args.seed = seed;
  args.wait_ns = wait_ns;
  args.drop_request = drop_request;
  args.prefetch_rows = 0;
  args.accept_len = accept_len;
  args.path_nodes = path_nodes;
  args.out_tokens = out_tokens;
  args.near_ties = near_ties;
  args.status = status;
  // Every host-side check has passed: nothing was enqueued before this point.
  if (clear_workspace &&
      cudaMemsetAsync(workspace, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  char *ws = static_cast<char *>(workspace);
  args.done = reinterpret_cast<uint32_t *>(ws);
  ws += align256(sizeof(uint32_t) * (B + 1));
  args.flags = reinterpret_cast<int32_t *>(ws);
  ws += align256(sizeof(int32_t) * T);
  args.fallback = reinterpret_cast<int32_t *>(ws);

  if (greedy) return launch_verify_greedy(args, static_cast<cudaStream_t>(stream));
  if (V <= kMaxCS * kRegChunk)
    return launch_verify_reg(args, (V + kRegChunk - 1) / kRegChunk, nucleus,
                             static_cast<cudaStream_t>(stream));
  const size_t smem = sizeof(float) * 2 * static_cast<size_t>(chunk);
  static std::atomic<size_t> granted[kMaxDevices];
  if (!allow_dynamic_smem(tree_verify_cluster_kernel, smem, granted)) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T) * CS, 1, 1);
  cfg.blockDim = dim3(kVThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attribute(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, tree_verify_cluster_kernel, args) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}
}  // namespace spec

extern "C" int spec_tree_verify(const float *target_logits, const float *draft_logits,
                                const int32_t *tokens, const int32_t *parents,
                                const int32_t *tree_offsets, int B, int T, int V,
                                float temperature, uint64_t seed, int32_t *accept_len,
                                int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties,
                                int max_depth_plus1, void *workspace, size_t workspace_bytes,
                                int32_t *status, void *stream) {
  return spec::verify_entry(target_logits, draft_logits, tokens, parents, tree_offsets, B, T, V,
                            temperature, 1.f, seed, accept_len, path_nodes, out_tokens, near_ties,
                            max_depth_plus1, workspace, workspace_bytes, status, stream, false);
}

extern "C" int spec_tree_verify_top_p(const float *target_logits, const float *draft_logits,
                                      const int32_t *tokens, const int32_t *parents,
                                      const int32_t *tree_offsets, int B, int T, int V,
                                      float temperature, float top_p, uint64_t seed,
                                      int32_t *accept_len, int32_t *path_nodes,
                                      int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                                      void *workspace, size_t workspace_bytes, int32_t *status,
                                      void *stream) {
  return spec::verify_entry(target_logits, draft_logits, tokens, parents, tree_offsets, B, T, V,
                            temperature, top_p, seed, accept_len, path_nodes, out_tokens, near_ties,
                            max_depth_plus1, workspace, workspace_bytes, status, stream, false);
}

extern "C" int spec_test_verify_timeout(const float *target_logits, const float *draft_logits,
                                        const int32_t *tokens, const int32_t *parents,
                                        const int32_t *tree_offsets, int B, int T, int V,
                                        float temperature, uint64_t seed, int32_t *accept_len,
                                        int32_t *path_nodes, int32_t *out_tokens,
                                        int32_t *near_ties, int max_depth_plus1, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream,
                                        uint64_t wait_ns, int drop_request) {
  // the register-resident stochastic kernel only, a short positive limit
  if (!(temperature > 0.f) || V > spec::kMaxCS * spec::kRegChunk) return SPEC_ERR_SHAPE;
  if (wait_ns == 0 || wait_ns > spec::kWaitLimitNs || drop_request < 0 || drop_request >= B)
    return SPEC_ERR_SHAPE;
  return spec::verify_entry(target_logits, draft_logits, tokens, parents, tree_offsets, B, T, V,
                            temperature, 1.f, seed, accept_len, path_nodes, out_tokens, near_ties,
                            max_depth_plus1, workspace, workspace_bytes, status, stream, false,
                            wait_ns, drop_request);
}
