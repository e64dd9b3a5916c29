// Steps V1-V4 and R: verification of a speculated token tree.  Stochastic
// verification runs one thread-block cluster per node (the node's target and
// draft rows split across the cluster's shared memory, about 16K entries per
// CTA); greedy verification runs the per-node kernel of verify_node.cu.
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
// group.  The last group of a request to finish then walks the tree in one
// warp.
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

// Per-CTA scratch for one reduction round, double buffered by round parity
// so a round never waits for the previous round's readers.
struct RoundScratch {
  float w[2][kVWarps][2];
  int wi[2][kVWarps];
};
static_assert(kVWarps == 32, "warp 0 combines one partial per lane");

// Cluster all-gather slots: every CTA pushes its partials into slot [rank]
// of every peer with remote stores, so after one cluster barrier all values
// are read from local shared memory.  Double buffered by round parity.
struct Gather {
  float v[2][kMaxCS][4];
};

// Barrier of one node's CTA group: the cluster barrier when the group spans
// several CTAs, else the CTA barrier.
__device__ __forceinline__ void group_sync(int CS) {
  if (CS > 1) cluster_sync_all();
  else __syncthreads();
}

// Publish this CTA's float4 to slot [rank] of every CTA of the group.
__device__ __forceinline__ void gather_put(Gather &gx, int parity, int rank, int CS, int lane,
                                           float4 val) {
  if (lane < CS) {
    if (CS > 1) st_peer_f32x4(peer_addr(&gx.v[parity][rank][0], lane), val);
    else *reinterpret_cast<float4 *>(&gx.v[parity][0][0]) = val;
  }
}

// Sum `x` over the CTA (warp shuffles, then warp 0 over the 32 warp
// partials) and over the group.  Returns the group total (identical in every
// CTA: partials are added in rank order) and, in `parts`, the per-CTA totals.
// One __syncthreads and one group barrier.
__device__ float cluster_round_sum(float x, RoundScratch &rs, Gather &gx, int parity, int rank,
                                   int CS, float *parts) {
  x = warp_sum(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) rs.w[parity][w][0] = x;
  __syncthreads();
  if (w == 0) {
    const float v = warp_sum(rs.w[parity][l][0]);
    gather_put(gx, parity, rank, CS, l, make_float4(v, 0.f, 0.f, 0.f));
  }
  group_sync(CS);
  float tot = 0.f;
  for (int r = 0; r < CS; ++r) {
    const float v = gx.v[parity][r][0];
    if (parts) parts[r] = v;
    tot += v;
  }
  return tot;
}

__global__ void __launch_bounds__(kVThreads)
tree_verify_cluster_kernel(const VerifyArgs a) {
  extern __shared__ __align__(128) float vsm[];  // [chunk] target side, [chunk] draft side
  __shared__ RoundScratch rs;
  __shared__ __align__(16) Gather gx;
  __shared__ TreeSmem ts;
  __shared__ int s_pick, s_pickw;
  __shared__ float s_cb[2], s_before;
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
    if (bulk && len > 0) {
      mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(len) * 4u);
      bulk_copy_g2s(lrow, trow_g + v0, static_cast<uint32_t>(len) * 4u, &bars[0]);
    }
  }
  const NodeCtx c = load_tree(a, t, ts);
  const int k = c.k;
  const bool need_draft = !c.err && !greedy && k > 0;
  if (tid == 0 && bulk && need_draft && len > 0) {
    mbar_arrive_expect_tx(&bars[1], static_cast<uint32_t>(len) * 4u);
    bulk_copy_g2s(drow, drow_g + v0, static_cast<uint32_t>(len) * 4u, &bars[1]);
  }
  load_children(a, c, t, ts);
  // ---- wait for the slices (a copy issued for a node is always waited for)
  bool timed_out = false;
  if (bulk && len > 0) {
    if (!mbar_wait(&bars[0], 0)) timed_out = true;
    if (need_draft && !mbar_wait(&bars[1], 0)) timed_out = true;
  } else if (!c.err) {
    for (int i = tid; i < len; i += kVThreads) {
      lrow[i] = __ldcs(trow_g + v0 + i);
      if (need_draft) drow[i] = __ldcs(drow_g + v0 + i);
    }
  }
  if (timed_out && tid == 0) report(a.status, c.b, SPEC_ERR_TIMEOUT);
  __syncthreads();

  if (!c.err) {
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
      if (w_id == 0) {
        const ArgMax r = warp_argmax(ArgMax{rs.w[0][lane][0], rs.wi[0][lane]});
        gather_put(gx, 0, rank, CS, lane, make_float4(r.v, __int_as_float(r.i), 0.f, 0.f));
      }
      group_sync(CS);
      if (rank == 0 && tid == 0) {
        ArgMax g{-INFINITY, 0x7fffffff};
        for (int r = 0; r < CS; ++r) g = better(g, ArgMax{gx.v[0][r][0], __float_as_int(gx.v[0][r][1])});
        a.fallback[t] = g.i;
        for (int j = 0; j < k; ++j) {
          const int ch = ts.child[j];
          a.flags[c.lo + ch] = (ts.tok[ch] == g.i) ? kFlagAccept : 0;
        }
      }
    } else {
      const float T_ = a.temp, iT = a.inv_temp;
      const float l2s = iT * 1.4426950408889634f;  // exp(x / T) = 2^(x * l2s)
      // ---- V1: per-thread max and sum of exp((x - m)/T) over the thread's
      //      elements, combined over the CTA and the cluster in one round
      float ml = -INFINITY, md = -INFINITY;
      for (int i = tid; i < len; i += kVThreads) {
        ml = fmaxf(ml, lrow[i]);
        if (need_draft) md = fmaxf(md, drow[i]);
      }
      float sl = 0.f, sd = 0.f;
      for (int i = tid; i < len; i += kVThreads) {
        const float el = fast_exp2((lrow[i] - ml) * l2s);
        lrow[i] = el;
        sl += el;
        if (need_draft) {
          const float ed = fast_exp2((drow[i] - md) * l2s);
          drow[i] = ed;
          sd += ed;
        }
      }
      // warp combine of (m, s) pairs
      const float wml = warp_max(ml), wmd = warp_max(md);
      const float wsl = warp_sum(sl > 0.f ? sl * fast_exp2((ml - wml) * l2s) : 0.f);
      const float wsd = warp_sum(sd > 0.f ? sd * fast_exp2((md - wmd) * l2s) : 0.f);
      __shared__ float s_pair[kVWarps][4];
      if (lane == 0) {
        s_pair[w_id][0] = wml;
        s_pair[w_id][1] = wsl;
        s_pair[w_id][2] = wmd;
        s_pair[w_id][3] = wsd;
      }
      __syncthreads();
      if (w_id == 0) {
        const float pm = s_pair[lane][0], ps = s_pair[lane][1];
        const float qm = s_pair[lane][2], qs = s_pair[lane][3];
        const float cm = warp_max(pm), cmd = warp_max(qm);
        const float cs = warp_sum(ps > 0.f ? ps * fast_exp2((pm - cm) * l2s) : 0.f);
        const float csd = warp_sum(qs > 0.f ? qs * fast_exp2((qm - cmd) * l2s) : 0.f);
        gather_put(gx, parity, rank, CS, lane, make_float4(cm, cs, cmd, csd));
      }
      group_sync(CS);
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
        kept[r] = part[r].y > 0.f ? part[r].y * fast_exp2((part[r].x - Ml) * l2s) : 0.f;
        Sp += kept[r];
        if (need_draft && part[r].w > 0.f) Sq += part[r].w * fast_exp2((part[r].z - Md) * l2s);
      }
      for (int r = 0; r < CS; ++r) kept[r] /= Sp;  // chunk sums of p
      parity ^= 1;
      // the children's p(x) and q(x), in parallel (read by the chain below)
      if (tid < k) {
        ts.cP[tid] = precise_prob(ts.cP[tid], Ml, T_, iT, Sp);
        ts.cQ[tid] = precise_prob(ts.cQ[tid], Md, T_, iT, Sq);
      }
      // p(v), q(v) for this thread's elements
      const float scale_l = ml == -INFINITY ? 0.f : fast_exp2((ml - Ml) * l2s) / Sp;
      const float scale_d = (need_draft && md != -INFINITY) ? fast_exp2((md - Md) * l2s) / Sq : 0.f;
      for (int i = tid; i < len; i += kVThreads) {
        lrow[i] *= scale_l;
        if (need_draft) drow[i] *= scale_d;
      }

      __syncthreads();  // the children's probabilities are in shared memory
      // ---- V2: the children's accept tests, one reduction per rejection
      float c_prev = 0.f, W_prev = 1.f;
      for (int j = 0; j < k; ++j) {
        const int ch = ts.child[j];
        const float P = ts.cP[j];
        const float Q = ts.cQ[j];
        const float alpha = Q > 0.f ? fminf(1.f, fmaxf(0.f, fmaf(-c_prev, Q, P)) / (W_prev * Q)) : 1.f;
        if (rank == 0 && tid == 0) {
          const float uu = ts.cU[j];
          int f = (uu < alpha) ? kFlagAccept : 0;
          if (fabsf(uu - alpha) < kTieBand) f |= kFlagTie;
          a.flags[c.lo + ch] = f;
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
      const float target = ts.ufb * total;
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
        if (w_id == 0) {
          // inclusive scan of the warp partials, first one passing the target
          const float v = rs.w[parity][lane][1];
          float inc = v;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
          }
          const uint32_t hit = __ballot_sync(0xffffffffu, prefix + inc > target);
          const int L = hit ? __ffs(hit) - 1 : -1;
          const float before_l = __shfl_sync(0xffffffffu, prefix + inc - v, L < 0 ? 0 : L);
          if (lane == 0) {
            s_pickw = L;
            s_before = before_l;
          }
        }
        __syncthreads();
        const int pick_w = s_pickw;
        const float before = s_before;
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
    group_sync(CS);  // no CTA leaves while a peer may still read its exchange slots
  } else if (rank == 0 && tid == 0 && c.b >= 0) {
    report(a.status, c.b, c.err);
  }
  if (rank == 0) arrive_and_walk(a, c, ts, gridDim.x / CS);
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

  if (greedy) return launch_verify_greedy(args, static_cast<cudaStream_t>(stream));
  const size_t smem = sizeof(float) * 2 * static_cast<size_t>(chunk);
  static int configured_smem = -1;
  if (configured_smem < static_cast<int>(smem)) {
    if (cudaFuncSetAttribute(tree_verify_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  if (cudaLaunchKernelEx(&cfg, tree_verify_cluster_kernel, args) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}
