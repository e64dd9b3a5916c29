// Steps V1-V4 and R for stochastic verification with the node's rows held in
// registers: one thread-block cluster of CS = ceil(V / 16384) CTAs per node,
// each CTA's 512 threads holding 32 entries of its slice of the target row
// and, for internal nodes, of the draft row.
//
// Sources: speculative-decoding explainer (intelliparadigm.com) §2.2
// 三阶段工作流程详解 — stage 2: accept probability alpha = min(1, p/q); stage 3:
// check left to right, stop at the first rejection and replace it with a new
// target prediction (output distribution equal to the target's).  SpecInfer
// developer article §2.1: the accept stage keeps the longest verified prefix.
//
// Layout.  Warp w of the CTA at cluster rank r owns the 1024 vocabulary
// entries [v0 + 1024 w, v0 + 1024 (w + 1)), v0 = 16384 r; lane l holds, for
// steps m = 0..7, the four entries v0 + 1024 w + 128 m + 4 l + (0..3).  The
// rows go from global memory straight into registers (coalesced 16-byte
// loads), and every pass over the vocabulary is a register loop: no shared
// memory traffic, and each warp's exponentials share the warp's own maximum,
// so no CTA barrier is needed before the group totals.
//
// Group totals.  Every warp pushes its partial into slot [rank][warp] of
// every CTA of the group with st.async; a round's mbarrier completes when all
// CS x 16 partials have landed, and every warp adds them in the same order,
// so all threads of the group hold bit-identical totals.
//
// The acceptance chain (residual in closed form, stop at the first accepted
// child) and the inverse-CDF draw follow the description in verify.cu.
#include "verify_common.cuh"

namespace spec {

namespace {

constexpr int kRThreads = 512;
constexpr int kRWarps = kRThreads / 32;
constexpr int kRVec = 8;                     // float4 per thread per row
constexpr int kRSpan = 32 * 4 * kRVec;       // vocabulary entries per warp
static_assert(kRWarps * kRSpan == kRegChunk, "CTA slice");

struct RegExchange {
  float4 stat[kMaxCS][kRWarps];     // per warp: max target logit, sum of target exps, same for draft
  float part[2][kMaxCS][kRWarps];   // reduction rounds, by round parity
  int last[kRWarps];                // rare path: per warp, its last entry of positive weight
};

// The node's scalars, computed once by the CTA's last warp: the children's
// p(x), q(x) and accept uniforms, and the fallback draw's uniform.
struct NodeScalars {
  float P[SPEC_MAX_TREE_NODES], Q[SPEC_MAX_TREE_NODES], U[SPEC_MAX_TREE_NODES];
  float u_fb;
  int near;                          // top-p: bit 0 (p) / 1 (q): an entry other than tau is near it
  int ctie[SPEC_MAX_TREE_NODES];     // top-p: child j's entry is near tau at such a node
};

// One CTA's candidates for tau after the first radix pass: the bits of its
// entries (p row, q row) whose top 8 bits equal tau's; n counts them all,
// also beyond the capacity (then the radix passes continue instead).
constexpr int kCandCap = 512;
struct __align__(16) TopPCands {
  uint32_t n[4];
  uint32_t v[2][kCandCap];
};

// Top-p working storage (dynamic shared memory).  Masses are fixed point,
// value * 2^40 rounded to u64, so histogram sums are exact and independent
// of the order of the atomic adds, and the rounding of a whole row stays
// below V * 2^-41 of its mass.
struct TopPSmem {
  // per warp: [row (p, q)][high, low 20 bits of the mass][digit]; a warp
  // adds at most 1024 entries of a row, so each half stays below 2^30
  uint32_t warp_hist[kRWarps][2][2][256];
  unsigned long long cta[2][2][256];               // the CTA's histogram, by pass parity
  unsigned long long recv[2][kMaxCS][2][256];      // every CTA's histogram, by pass parity
  unsigned long long hsum[2][256];                 // the group's histogram
  unsigned long long state[2][4];   // per row: prefix bits, mass above, digit mass, target
  float2 statp[kMaxCS][kRWarps];    // per warp: its mass of the filtered p, near flags
  TopPCands cand_local;             // this CTA's candidates
  TopPCands cand_recv[kMaxCS];      // every CTA's candidates
  uint64_t bar[2], sbar, gbar;
};
constexpr uint32_t kHistBytes = 2 * 256 * 8;  // one CTA histogram
constexpr float kFixedScale = 1099511627776.f;  // 2^40
// Entries other than tau within this many ulps of it may be ordered the
// other way round in exact arithmetic (the exponentials' rounding).
constexpr int kTauUlps = 128;

__device__ __forceinline__ unsigned long long fixed_mass(float v) {
  return __float2ull_rn(v * kFixedScale);
}
// hist[bin] += fixed_mass(v), split into its bits 20 and up (at saddr) and
// its low 20 bits (at saddr + 1 KB), 32-bit shared-memory adds (a 64-bit
// shared add measured about twice as slow; an add of zero is skipped, as
// the first is for most entries: p < 2^-20), as one unit: the scaling, the
// conversion and the adds stay together, so that an unrolled loop over a
// thread's entries does not hold all their conversions in registers at once.
__device__ __forceinline__ void hist_add(uint32_t saddr, float v) {
  asm volatile(
      "{\n\t.reg .f32 s;\n\t.reg .u64 m;\n\t.reg .u32 hi, lo;\n\t.reg .pred big;\n\t"
      "mul.rn.f32 s, %1, 0f53800000;\n\t"   // v * 2^40 (exact)
      "cvt.rni.u64.f32 m, s;\n\t"
      "cvt.u32.u64 lo, m;\n\t"
      "shr.u64 m, m, 20;\n\t"
      "cvt.u32.u64 hi, m;\n\t"
      "and.b32 lo, lo, 1048575;\n\t"
      "setp.ne.u32 big, hi, 0;\n\t"
      "@big red.shared.add.u32 [%0], hi;\n\t"
      "setp.ne.u32 big, lo, 0;\n\t"
      "@big red.shared.add.u32 [%0+1024], lo;\n\t}"
      :
      : "r"(saddr), "f"(v)
      : "memory");
}

// The radix digits of tau's bits (non-negative floats: bit 31 is 0): the
// exponent, then 8, 8 and 7 bits of the mantissa.
__device__ __forceinline__ int radix_shift(int pass) { return pass == 0 ? 23 : (pass == 1 ? 15 : (pass == 2 ? 7 : 0)); }
__device__ __forceinline__ uint32_t radix_mask(int pass) { return pass == 3 ? 127u : 255u; }
__device__ __forceinline__ int radix_top(int pass) { return pass == 0 ? 31 : radix_shift(pass - 1); }
__device__ __forceinline__ bool near_bits(uint32_t x, uint32_t t) {
  const int d = static_cast<int>(x - t);
  return d >= -kTauUlps && d <= kTauUlps;
}
constexpr int kScalarWarp = kRWarps - 1;

// 32 entries of a row into registers; entries at or past `end` read as -inf.
__device__ __forceinline__ void load_row(const float *row, int base, int end, bool vec,
                                         float4 (&x)[kRVec]) {
#pragma unroll
  for (int m = 0; m < kRVec; ++m) {
    const int i = base + 128 * m;
    if (vec && i + 3 < end) {
      x[m] = __ldcs(reinterpret_cast<const float4 *>(row + i));
    } else {
      x[m].x = i < end ? __ldcs(row + i) : -INFINITY;
      x[m].y = i + 1 < end ? __ldcs(row + i + 1) : -INFINITY;
      x[m].z = i + 2 < end ? __ldcs(row + i + 2) : -INFINITY;
      x[m].w = i + 3 < end ? __ldcs(row + i + 3) : -INFINITY;
    }
  }
}

__device__ __forceinline__ float max4(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }

// The residual weight of one entry: max(0, p - c q), or p while c == 0.
__device__ __forceinline__ float resid(float p, float q, float c) {
  return c != 0.f ? fmaxf(0.f, fmaf(-c, q, p)) : p;
}

// The residual weight of a thread's entries for c > 0 (every rejection
// round): the sum of max(0, p - c q) without the c == 0 case, with paired
// fp32 FMAs and a paired accumulator (two partial sums, added at the end).
__device__ __forceinline__ float resid_sum_pos(const float4 (&p)[kRVec], const float4 (&q)[kRVec],
                                               float c) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int m = 0; m < kRVec; ++m) {
    asm("{\n\t.reg .b64 nc, q01, q23, p01, p23, r01, r23, acc;\n\t"
        ".reg .f32 r0, r1, r2, r3;\n\t"
        "mov.b64 nc, {%2, %2};\n\t"
        "mov.b64 q01, {%3, %4};\n\t"
        "mov.b64 q23, {%5, %6};\n\t"
        "mov.b64 p01, {%7, %8};\n\t"
        "mov.b64 p23, {%9, %10};\n\t"
        "fma.rn.f32x2 r01, nc, q01, p01;\n\t"
        "fma.rn.f32x2 r23, nc, q23, p23;\n\t"
        "mov.b64 {r0, r1}, r01;\n\t"
        "mov.b64 {r2, r3}, r23;\n\t"
        "max.f32 r0, r0, 0f00000000;\n\t"
        "max.f32 r1, r1, 0f00000000;\n\t"
        "max.f32 r2, r2, 0f00000000;\n\t"
        "max.f32 r3, r3, 0f00000000;\n\t"
        "mov.b64 r01, {r0, r1};\n\t"
        "mov.b64 r23, {r2, r3};\n\t"
        "mov.b64 acc, {%0, %1};\n\t"
        "add.rn.f32x2 acc, acc, r01;\n\t"
        "add.rn.f32x2 acc, acc, r23;\n\t"
        "mov.b64 {%0, %1}, acc;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(-c), "f"(q[m].x), "f"(q[m].y), "f"(q[m].z), "f"(q[m].w), "f"(p[m].x), "f"(p[m].y),
          "f"(p[m].z), "f"(p[m].w));
  }
  return a0 + a1;
}

__device__ __forceinline__ float sum4_resid(float4 p, float4 q, float c) {
  return (resid(p.x, q.x, c) + resid(p.y, q.y, c)) + (resid(p.z, q.z, c) + resid(p.w, q.w, c));
}

__device__ __forceinline__ float pick4(const float4 v, int c) {
  return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

// The warp totals of the eight steps' values ls[0..7] at once: a transposed
// butterfly (each exchange halves the values a lane carries) leaves step m's
// total in lanes 4m .. 4m+3 and returns it there.  Every total adds the same
// pairs in the same order as warp_sum, so it is bit-identical to it.
__device__ __forceinline__ float step_totals(const float (&ls)[kRVec], int lane) {
  static_assert(kRVec == 8, "three halving exchanges");
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float v4[4], v2[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? ls[4 + i] : ls[i];
    const float give = b4 ? ls[i] : ls[4 + i];
    v4[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? v4[2 + i] : v4[i];
    const float give = b3 ? v4[i] : v4[2 + i];
    v2[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
  }
  float v = (b2 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? v2[0] : v2[1], 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

__device__ __forceinline__ float warp_scan(float v, int lane) {  // inclusive
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

}  // namespace

template <bool TOPP>
__global__ void __launch_bounds__(kRThreads, 1)
tree_verify_reg_kernel(const VerifyArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];   // TopPSmem when TOPP
  __shared__ __align__(16) RegExchange ex;
  __shared__ TreeSmem ts;
  __shared__ NodeScalars ns;
  __shared__ __align__(8) uint64_t xbar[3];   // exchange: statistics round, rounds by parity
  __shared__ __align__(8) uint64_t nbar;      // the node's scalars are in `ns`

  const int CS = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_rank());
  const int t = blockIdx.x / CS;
  const int tid = threadIdx.x, w_id = tid >> 5, lane = tid & 31;
  const int v0 = rank * kRegChunk;
  const int end = min(a.V, v0 + kRegChunk);     // this CTA's slice is [v0, end)
  const int base = v0 + w_id * kRSpan + 4 * lane;
  const bool vec = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0) &&
                   ((reinterpret_cast<uintptr_t>(a.draft) & 15) == 0);
  const float *trow = a.target + static_cast<size_t>(t) * a.V;
  const float *drow = a.draft + static_cast<size_t>(t) * a.V;

  pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&xbar[i], 1);
    mbar_init(&nbar, 1);
    if constexpr (TOPP) {
      TopPSmem &tp = *reinterpret_cast<TopPSmem *>(dyn_smem);
      mbar_init(&tp.bar[0], 1);
      mbar_init(&tp.bar[1], 1);
      mbar_init(&tp.sbar, 1);
      mbar_init(&tp.gbar, 1);
    }
    fence_barrier_init();
  }
  pdl_wait();
  // the tree first, then the target row
  const TreeLoads tl = tree_loads(a, t);
  float4 xp[kRVec], xq[kRVec];
  if constexpr (TOPP) {
    load_row(trow, base, end, vec, xp);
  } else if (a.prefetch_rows && tid == 0 && vec && end > v0) {
    // the slice goes to L2 at once, before the node knows whether it is a
    // leaf (whose row is read only if the walk ends there); only when every
    // CTA of the launch is resident, since a leaf's prefetch otherwise takes
    // bandwidth from the nodes still running
    const uint32_t bytes = (static_cast<uint32_t>(end - v0) * 4u) & ~15u;
    if (bytes > 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       reinterpret_cast<uint64_t>(trow + v0)),
                   "r"(bytes)
                   : "memory");
  }
  if (CS > 1) cluster_arrive_relaxed();   // waited for before the first remote store
  const NodeCtx ca = load_tree_a(a, t, ts, tl);
  // Internal nodes only: the draft row is requested as soon as the staged
  // window shows a child, before the tree is validated.
  const bool early_draft = has_children(ca, t, ts);
  if constexpr (!TOPP) {
    if (!early_draft && !ca.err && ca.u != 0) {
      // A leaf other than a lone root: its only result is the token drawn if
      // the walk accepts the path down to it, which the walker then draws
      // itself.  The leaf arrives and frees its SMs.
      stage_request(ca, t, ts);
      if (CS > 1) cluster_wait();
      if (rank == 0) arrive_and_walk(a, ca, ts, -1, 0, false, true);
      return;
    }
    load_row(trow, base, end, vec, xp);
  }
  if (early_draft) {
    load_row(drow, base, end, vec, xq);
  } else {
#pragma unroll
    for (int m = 0; m < kRVec; ++m) xq[m] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const NodeCtx c = load_tree_b(a, t, ts, ca);
  const int k = c.k;
  const bool need_draft = !c.err && k > 0;   // leaves never read their draft row
  // the root: whether the request's deepest path fits the output rows, while
  // the rows are in flight (its early arrival needs it)
  if (!c.err && c.u == 0 && w_id == 0) {
    const bool f = path_fits_quiet(a, c.n, ts.par);
    if (lane == 0) ts.fits = f ? 1 : 0;
  }
  if (need_draft && !early_draft) load_row(drow, base, end, vec, xq);   // not expected
  // The scalar warp draws the node's uniforms (children's accept tests, the
  // fallback draw) and reads the children's raw logits while the rows are in
  // flight; lane j handles child j (and lane k the fallback draw's uniform).
  const bool scalar_warp = w_id == kScalarWarp;
  float rawP[4], rawQ[4];
  if (scalar_warp && !c.err) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int j = lane + 32 * s;
      rawP[s] = rawQ[s] = 0.f;
      if (j < k) {
        const int ch = ts.child[j];
        const int x = ts.tok[ch];
        if (in_bounds(x, a.V, a.status, c.b)) {
          rawP[s] = __ldg(trow + x);
          rawQ[s] = __ldg(drow + x);
        }
        ns.U[j] = spec_uniform(a.seed, ch, c.b, 0);
      } else if (j == k) {
        ns.u_fb = spec_uniform(a.seed, c.u, c.b, 1);
      }
    }
  }
  if (tid == 0 && !c.err) mbar_arrive_expect_tx(&xbar[0], static_cast<uint32_t>(CS * kRWarps * 16));
  if (CS > 1) cluster_wait();  // every CTA of the group is running

  bool ok = true;
  int stop = k;        // first accepted child, k when every child is rejected
  int my_flag = 0;     // thread j < k: the flag of child j
  int p_ok = -1;       // parity of the last reduction round that moved the residual
  float slice_lo = 0.f, slice_hi = 0.f;   // that round's two slice totals (two CTAs)
  int near = 0;            // top-p: ns.near
  uint32_t tau_kept[2] = {0u, 0u};   // top-p: tau of p and q after renormalisation
  float c_prev = 0.f, Ml = 0.f, Sp = 1.f;
  const float l2s = a.inv_temp * 1.4426950408889634f;  // exp(x / T) = 2^(x * l2s)
  if (!c.err) {
    // ---- V1: the warp's maxima, exponentials in place, the warp's sums.
    //      The target row first: the draft row was requested later, so its
    //      loads are still in flight while the target's work runs.
    // half of the exponentials on the MUFU pipe, half on the FMA pipe
    auto expo = [&](float v, float nb, int m) -> float {
      const float z = fmaf(v, l2s, nb);
      return m < kRVec / 2 ? fast_exp2(z) : exp2_taylor(z);
    };
    float ml = -INFINITY;
#pragma unroll
    for (int m = 0; m < kRVec; ++m) ml = fmaxf(ml, max4(xp[m]));
    ml = warp_max(ml);
    const float nl = ml == -INFINITY ? 0.f : -ml * l2s;
    float sl = 0.f;
#pragma unroll
    for (int m = 0; m < kRVec; ++m) {
      xp[m].x = expo(xp[m].x, nl, m);
      xp[m].y = expo(xp[m].y, nl, m);
      xp[m].z = expo(xp[m].z, nl, m);
      xp[m].w = expo(xp[m].w, nl, m);
      sl += (xp[m].x + xp[m].y) + (xp[m].z + xp[m].w);
    }
    float md = -INFINITY;
#pragma unroll
    for (int m = 0; m < kRVec; ++m) md = fmaxf(md, max4(xq[m]));
    md = need_draft ? warp_max(md) : -INFINITY;
    const float nd = md == -INFINITY ? 0.f : -md * l2s;
    float sd = 0.f;
    if (need_draft) {
#pragma unroll
      for (int m = 0; m < kRVec; ++m) {
        xq[m].x = expo(xq[m].x, nd, m);
        xq[m].y = expo(xq[m].y, nd, m);
        xq[m].z = expo(xq[m].z, nd, m);
        xq[m].w = expo(xq[m].w, nd, m);
        sd += (xq[m].x + xq[m].y) + (xq[m].z + xq[m].w);
      }
    }
    sl = warp_sum(sl);
    sd = warp_sum(sd);
    // (the failure test withholds the last CTA's share for one request, so
    // that every CTA's wait on this exchange runs out)
    if (lane < CS && !(c.b == a.drop_request && rank == CS - 1))
      st_async_v4_f32(peer_addr(&ex.stat[rank][w_id], lane), make_float4(ml, sl, md, sd),
                      peer_addr(&xbar[0], lane));
    if (!mbar_wait_for(&xbar[0], 0, a.wait_ns)) ok = false;
    // group maxima and sums, added in the same order by every warp
    const int nslot = CS * kRWarps;
    const float4 *flat = &ex.stat[0][0];
    float4 e[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = lane + 32 * s;
      e[s] = i < nslot ? flat[i] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    }
    float Mx = -INFINITY, Mdx = -INFINITY;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      Mx = fmaxf(Mx, e[s].x);
      Mdx = fmaxf(Mdx, e[s].z);
    }
    Ml = warp_max(Mx);
    const float Md = warp_max(Mdx);
    float sp = 0.f, sq = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (e[s].y > 0.f) sp += e[s].y * fast_exp2((e[s].x - Ml) * l2s);
      if (need_draft && e[s].w > 0.f) sq += e[s].w * fast_exp2((e[s].z - Md) * l2s);
    }
    Sp = warp_sum(sp);
    const float Sq = warp_sum(sq);
    // this warp's entries become p and q
    const float inv_sp = 1.f / Sp;
    const float inv_sq = need_draft ? 1.f / Sq : 0.f;
    const float sc_l = ml == -INFINITY ? 0.f : fast_exp2((ml - Ml) * l2s) * inv_sp;
    const float sc_d = (need_draft && md != -INFINITY) ? fast_exp2((md - Md) * l2s) * inv_sq : 0.f;
    // The children's p and q from their raw logits (scalar warp), published
    // with the uniforms through an mbarrier (release / acquire).  Without a
    // nucleus this needs only the group statistics, so the scalar warp does it
    // before scaling its own entries, and the accept tests wait less.
    uint32_t tau_bits[2] = {0u, 0u};
    float inv_nuc[2] = {1.f, 1.f};
    auto publish_children = [&]() {
      int nb = 0;
      if constexpr (TOPP) {
        const TopPSmem &tp = *reinterpret_cast<const TopPSmem *>(dyn_smem);
        for (int i = lane; i < CS * kRWarps; i += 32) nb |= static_cast<int>((&tp.statp[0][0])[i].y);
        nb = __reduce_or_sync(0xffffffffu, static_cast<unsigned>(nb));
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int j = lane + 32 * s;
        if (j < k) {
          float P = precise_prob(rawP[s], Ml, a.temp, a.inv_temp, 1.f) * inv_sp;
          float Q = precise_prob(rawQ[s], Md, a.temp, a.inv_temp, 1.f) * inv_sq;
          if constexpr (TOPP) {
            // Membership follows the child's own entry of the filtered rows:
            // the same operations on the same operands as its owner thread
            // (warp maximum from the exchanged statistics, the same exp path).
            const int x = ts.tok[ts.child[j]];
            const int r = x / kRegChunk, off = x - r * kRegChunk;
            const int wo = off / kRSpan, mo = (off % kRSpan) >> 7;
            const float4 st = ex.stat[r][wo];
            const float zp = fmaf(rawP[s], l2s, -st.x * l2s), zq = fmaf(rawQ[s], l2s, -st.z * l2s);
            const float eP = (mo < kRVec / 2 ? fast_exp2(zp) : exp2_taylor(zp)) *
                             (fast_exp2((st.x - Ml) * l2s) * inv_sp);
            const float eQ = (mo < kRVec / 2 ? fast_exp2(zq) : exp2_taylor(zq)) *
                             (fast_exp2((st.z - Md) * l2s) * inv_sq);
            P = __float_as_uint(eP) >= tau_bits[0] ? P * inv_nuc[0] : 0.f;
            Q = __float_as_uint(eQ) >= tau_bits[1] ? Q * inv_nuc[1] : 0.f;
            ns.ctie[j] = ((nb & 1) && near_bits(__float_as_uint(eP), tau_bits[0])) ||
                         ((nb & 2) && near_bits(__float_as_uint(eQ), tau_bits[1]));
          }
          ns.P[j] = P;
          ns.Q[j] = Q;
        }
      }
      if (lane == 0) ns.near = nb;
      __syncwarp();
      if (lane == 0) mbar_arrive(&nbar);
    };
    if constexpr (!TOPP) {
      if (scalar_warp) publish_children();
    }
#pragma unroll
    for (int m = 0; m < kRVec; ++m) {
      xp[m].x *= sc_l; xp[m].y *= sc_l; xp[m].z *= sc_l; xp[m].w *= sc_l;
      xq[m].x *= sc_d; xq[m].y *= sc_d; xq[m].z *= sc_d; xq[m].w *= sc_d;
    }
    // ---- top-p: the nucleus of p and of q.  tau is the largest entry whose
    //      upper tail {x >= tau} holds at least top_p of the mass; entries of
    //      that tail keep their mass, renormalised, the rest drop to 0.  The
    //      float bits of non-negative entries order like the values, so tau
    //      is found by radix passes over them (the exponent, then 8, 8 and 7
    //      mantissa bits): each pass sums the fixed-point mass of the entries
    //      still in play per digit and keeps the digit where the running mass
    //      from the top reaches top_p.  The first pass takes per-warp
    //      histograms, a CTA histogram and the group's by bulk copy; the
    //      entries sharing tau's exponent are then gathered from the group,
    //      and the other passes run on them in every CTA.
    if constexpr (TOPP) {
      TopPSmem &tp = *reinterpret_cast<TopPSmem *>(dyn_smem);
      // state[r] = {prefix bits of tau, mass above the prefix's digit range,
      // mass of the kept digit, target}; rows p (0) and q (1)
      if (tid < 8) (&tp.state[0][0])[tid] = 0ull;
      if (tid < 4) tp.cand_local.n[tid] = 0u;
      __syncthreads();
      // Warp r (rows p, q) finds the digit of row r, at bits [shift, shift + width)
      // of tau, where the running mass of tp.hsum from the top reaches the
      // target, and extends tp.state[r].
      auto find_digit = [&](int pass, int shift) {
        if (w_id < (need_draft ? 2 : 1)) {
          // warp r: the digit of row r where the running mass from the top
          // reaches the target (lane l holds digits 255 - 8l .. 248 - 8l)
          const int r = w_id;
          const unsigned long long *hr = &tp.hsum[r][0];
          unsigned long long lsum = 0ull;
#pragma unroll
          for (int i = 0; i < 8; ++i) lsum += hr[255 - 8 * lane - i];
          unsigned long long inc = lsum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
          }
          const unsigned long long prefix = tp.state[r][0], above = tp.state[r][1];
          unsigned long long target = tp.state[r][3];
          if (pass == 0) {
            // rounding may leave the row's total below top_p (then all is
            // kept); a top_p below the fixed-point unit keeps the top entry
            const unsigned long long total = __shfl_sync(0xffffffffu, inc, 31);
            target = max(1ull, min(fixed_mass(a.top_p), total));
          }
          const uint32_t hm = __ballot_sync(0xffffffffu, above + inc >= target);
          const int L = hm ? __ffs(hm) - 1 : 31;
          if (lane == L) {
            // the crossing digit; without one (an all-zero row) the lowest
            unsigned long long run = above + inc - lsum, new_above = above, dmass = 0ull;
            int digit = 0;
            bool found = false;
            for (int i = 0; i < 8 && !found; ++i) {
              const unsigned long long h = hr[255 - 8 * lane - i];
              if (run + h >= target || (hm == 0u && i == 7)) {
                found = true;
                digit = 255 - 8 * lane - i;
                new_above = run;
                dmass = h;
              }
              run += h;
            }
            tp.state[r][0] = prefix | (static_cast<unsigned long long>(digit) << shift);
            tp.state[r][1] = new_above;
            tp.state[r][2] = dmass;
            tp.state[r][3] = target;
          }
        }
      };
      auto gather_candidates = [&]() -> bool {
        TopPCands &cl = tp.cand_local;
        const uint32_t d0p = static_cast<uint32_t>(tp.state[0][0]) >> 23;
        const uint32_t d0q = need_draft ? static_cast<uint32_t>(tp.state[1][0]) >> 23 : 0xffffffffu;
        // this thread's entries in the digit, as bit masks over its 32 slots
        uint32_t mp = 0u, mq = 0u;
#pragma unroll
        for (int m = 0; m < kRVec; ++m)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint32_t bp = __float_as_uint(pick4(xp[m], cc));
            const uint32_t bq = __float_as_uint(pick4(xq[m], cc));
            mp |= (bp != 0u && (bp >> 23) == d0p) ? (1u << (4 * m + cc)) : 0u;
            mq |= (bq != 0u && (bq >> 23) == d0q) ? (1u << (4 * m + cc)) : 0u;
          }
        // a warp prefix of the counts, one atomic per warp and row
        auto slot_base = [&](int cnt, uint32_t *counter) -> int {
          int inc = cnt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
          }
          int base = 0;
          if (lane == 31 && inc > 0) base = static_cast<int>(atomicAdd(counter, static_cast<uint32_t>(inc)));
          return __shfl_sync(0xffffffffu, base, 31) + inc - cnt;
        };
        int atp = slot_base(__popc(mp), &cl.n[0]);
        int atq = slot_base(__popc(mq), &cl.n[1]);
#pragma unroll
        for (int m = 0; m < kRVec; ++m)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            if ((mp >> (4 * m + cc)) & 1u) {
              if (atp < kCandCap) cl.v[0][atp] = __float_as_uint(pick4(xp[m], cc));
              ++atp;
            }
            if ((mq >> (4 * m + cc)) & 1u) {
              if (atq < kCandCap) cl.v[1][atq] = __float_as_uint(pick4(xq[m], cc));
              ++atq;
            }
          }
        // (generic writes, read by the bulk copies)
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ok) {   // (no arrival after a wait ran out)
          mbar_arrive_expect_tx(&tp.gbar, static_cast<uint32_t>(CS * sizeof(TopPCands)));
          for (int r = 0; r < CS; ++r)
            bulk_copy_s2s(peer_addr(&tp.cand_recv[rank], r), smem_addr(&cl),
                          static_cast<uint32_t>(sizeof(TopPCands)), peer_addr(&tp.gbar, r));
        }
        if (ok && !mbar_wait_for(&tp.gbar, 0, a.wait_ns)) ok = false;
        // every CTA sees the same counts, so every CTA takes the same path
        // (and a CTA whose wait ran out takes one path, by the barrier)
        bool fits = ok;
        for (int r = 0; r < CS; ++r) fits = fits && tp.cand_recv[r].n[0] <= kCandCap &&
                                        tp.cand_recv[r].n[1] <= kCandCap;
        if (!__syncthreads_and(fits)) return false;
        // passes 1-3 on the candidates: the group histogram of the entries
        // still in play, from the candidates alone
        for (int lp = 1; lp < 4; ++lp) {
          const int shift = radix_shift(lp), top = radix_top(lp);
          const uint32_t dmask = radix_mask(lp);
          (&tp.hsum[0][0])[tid] = 0ull;   // 512 threads: 2 rows x 256 digits
          __syncthreads();
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            if (r == 1 && !need_draft) break;
            const uint32_t hi = static_cast<uint32_t>(tp.state[r][0]) >> top;
            for (int r2 = 0; r2 < CS; ++r2) {
              const int n = static_cast<int>(tp.cand_recv[r2].n[r]);
              for (int i = tid; i < n; i += kRThreads) {
                const uint32_t bits = tp.cand_recv[r2].v[r][i];
                if ((bits >> top) == hi)
                  atomicAdd(&tp.hsum[r][(bits >> shift) & dmask], fixed_mass(__uint_as_float(bits)));
              }
            }
          }
          __syncthreads();
          find_digit(lp, shift);
          __syncthreads();
        }
        return true;
      };
      for (int pass = 0; pass < 4; ++pass) {
        // After pass 0, tau's exponent is known, and few entries share it:
        // they are gathered from every CTA of the group in one exchange, and
        // passes 1-3 run on them locally (the same sums over the same
        // entries, so the same tau); too many, and the passes below run.
        if (pass == 1 && gather_candidates()) break;
        const int shift = radix_shift(pass), top = radix_top(pass);
        const uint32_t dmask = radix_mask(pass);
        const int par = pass & 1;
        const uint32_t hi_p = static_cast<uint32_t>(tp.state[0][0]) >> top;
        const uint32_t hi_q = static_cast<uint32_t>(tp.state[1][0]) >> top;
        uint32_t *wh = &tp.warp_hist[w_id][0][0][0];
        const uint32_t wh_addr = smem_addr(wh);
        for (int i = lane; i < 1024; i += 32) wh[i] = 0u;
        __syncwarp();
#pragma unroll
        for (int m = 0; m < kRVec; ++m) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const float v = pick4(xp[m], cc);
            const uint32_t bits = __float_as_uint(v);
            if (bits != 0u && (pass == 0 || (bits >> top) == hi_p))
              hist_add(wh_addr + 4u * ((bits >> shift) & dmask), v);
          }
        }
        if (need_draft) {
#pragma unroll
          for (int m = 0; m < kRVec; ++m) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const float v = pick4(xq[m], cc);
              const uint32_t bits = __float_as_uint(v);
              if (bits != 0u && (pass == 0 || (bits >> top) == hi_q))
                hist_add(wh_addr + 2048u + 4u * ((bits >> shift) & dmask), v);
            }
          }
        }
        __syncthreads();
        {
          const int row = tid >> 8, bin = tid & 255;   // 512 threads: 2 rows x 256 digits
          unsigned long long h = 0ull;
#pragma unroll
          for (int ww = 0; ww < kRWarps; ++ww)
            h += (static_cast<unsigned long long>(tp.warp_hist[ww][row][0][bin]) << 20) +
                 tp.warp_hist[ww][row][1][bin];
          tp.cta[par][row][bin] = h;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ok) {   // (no arrival after a wait ran out, as in the rounds below)
          mbar_arrive_expect_tx(&tp.bar[par], static_cast<uint32_t>(CS) * kHistBytes);
          for (int r = 0; r < CS; ++r)
            bulk_copy_s2s(peer_addr(&tp.recv[par][rank][0][0], r), smem_addr(&tp.cta[par][0][0]),
                          kHistBytes, peer_addr(&tp.bar[par], r));
        }
        if (ok && !mbar_wait_for(&tp.bar[par], (pass >> 1) & 1, a.wait_ns)) ok = false;
        {
          const int row = tid >> 8, bin = tid & 255;
          unsigned long long h = 0ull;
          for (int r = 0; r < CS; ++r) h += tp.recv[par][r][row][bin];
          tp.hsum[row][bin] = h;
        }
        __syncthreads();
        find_digit(pass, shift);
        __syncthreads();
      }
      // the nucleus: entries whose bits are >= tau's, renormalised.  An
      // entry other than tau within kTauUlps of it may sit on the other side
      // of tau in exact arithmetic: the node records that it has one, and
      // decisions that involve an entry near tau count as near-ties.
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const unsigned long long ge = tp.state[r][1] + tp.state[r][2];
        tau_bits[r] = static_cast<uint32_t>(tp.state[r][0]);
        inv_nuc[r] = ge > 0ull ? kFixedScale / static_cast<float>(ge) : 0.f;
        tau_kept[r] = __float_as_uint(__uint_as_float(tau_bits[r]) * inv_nuc[r]);
      }
      bool near_p = false, near_q = false;
      auto keep = [&](float v, int r, bool &nr) -> float {
        const uint32_t bits = __float_as_uint(v);
        nr |= bits != tau_bits[r] && near_bits(bits, tau_bits[r]);
        return bits >= tau_bits[r] ? v * inv_nuc[r] : 0.f;
      };
#pragma unroll
      for (int m = 0; m < kRVec; ++m) {
        xp[m].x = keep(xp[m].x, 0, near_p);
        xp[m].y = keep(xp[m].y, 0, near_p);
        xp[m].z = keep(xp[m].z, 0, near_p);
        xp[m].w = keep(xp[m].w, 0, near_p);
        if (need_draft) {
          xq[m].x = keep(xq[m].x, 1, near_q);
          xq[m].y = keep(xq[m].y, 1, near_q);
          xq[m].z = keep(xq[m].z, 1, near_q);
          xq[m].w = keep(xq[m].w, 1, near_q);
        }
      }
      // every warp's mass of the filtered p and its near flag, to every CTA
      float sf = 0.f;
#pragma unroll
      for (int m = 0; m < kRVec; ++m) sf += (xp[m].x + xp[m].y) + (xp[m].z + xp[m].w);
      sf = warp_sum(sf);
      const float nflags = (__any_sync(0xffffffffu, near_p) ? 1.f : 0.f) +
                           (__any_sync(0xffffffffu, near_q) ? 2.f : 0.f);
      if (tid == 0) mbar_arrive_expect_tx(&tp.sbar, static_cast<uint32_t>(CS * kRWarps * 8));
      if (lane < CS)
        st_async_v2_f32(peer_addr(&tp.statp[rank][w_id].x, lane), sf, nflags,
                        peer_addr(&tp.sbar, lane));
      if (ok && !mbar_wait_for(&tp.sbar, 0, a.wait_ns)) ok = false;
    }
    // top-p: the children's p and q need the nuclei
    if constexpr (TOPP) {
      if (scalar_warp) publish_children();
    }
    if (ok && !mbar_wait_for(&nbar, 0, a.wait_ns)) ok = false;
    if (TOPP) near = ns.near;

    // ---- V2: the children's accept tests in index order, stopping at the
    //      first accepted child (the walk never looks past it).  The test
    //      u < min(1, num / den) is taken as u * den < num, without a division.
    float W_prev = 1.f;
    bool frozen = false;   // a residual that summed to zero stays as it is
    int rounds = 0;
    // (slice_lo, slice_hi: the two CTAs' totals of the last round that moved the residual)
    for (int j = 0; j < k; ++j) {
      const float P = ns.P[j];
      const float Q = ns.Q[j];
      const float U = ns.U[j];
      bool accept, tie;
      const float num = fmaxf(0.f, fmaf(-c_prev, Q, P));
      const float den = W_prev * Q;
      if (Q > 0.f && num < den) {
        const float d = fmaf(U, den, -num);
        accept = d < 0.f;
        tie = fabsf(d) < kTieBand * den;
      } else {  // alpha = 1
        accept = true;
        tie = 1.f - U < kTieBand;
      }
      if (TOPP) tie |= ns.ctie[j] != 0;
      if (tid == j) my_flag = (accept ? kFlagAccept : 0) | (tie ? kFlagTie : 0);
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
      float wsum = resid_sum_pos(xp, xq, c_new);   // c_new > 0
      wsum = warp_sum(wsum);
      const int p = rounds & 1;
      if (tid == 0) mbar_arrive_expect_tx(&xbar[1 + p], static_cast<uint32_t>(CS * kRWarps * 4));
      if (lane < CS)
        st_async_f32(peer_addr(&ex.part[p][rank][w_id], lane), wsum, peer_addr(&xbar[1 + p], lane));
      if (ok && !mbar_wait_for(&xbar[1 + p], (rounds >> 1) & 1, a.wait_ns)) ok = false;
      ++rounds;
      const float *fl = &ex.part[p][0][0];
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int i = lane + 32 * s;
        if (i < nslot) acc += fl[i];
      }
      // the group total, each 16-lane half summed first: with two CTAs the
      // halves are the CTAs' slice totals, which the draw then reuses
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      const float Wn = acc + __shfl_xor_sync(0xffffffffu, acc, 16);
      if (Wn > 0.f) {
        c_prev = c_new;
        W_prev = Wn;
        p_ok = p;
        slice_lo = __shfl_sync(0xffffffffu, acc, 0);
        slice_hi = __shfl_sync(0xffffffffu, acc, 16);
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
  // A wait that ran out anywhere in the CTA: its threads may have taken
  // different decisions (a thread whose wait ran out skips the later waits
  // and may read the node's scalars before they are written), so the CTA
  // takes one path from here on: no draw, no published decision, and rank 0
  // arrives with the error bit.  Without a timeout every thread holds the
  // same decisions and the draw's barriers are met by all of them.
  const bool cta_timeout = __syncthreads_or(!ok);

  int writer = 0;  // the CTA of the group that publishes the node's results
  RootArrival early{false, 0u};
  if (!c.err && !cta_timeout) {
    // ---- V3: when every child is rejected (or u is a leaf), the token
    //      emitted on stopping here: inverse CDF of r ∝ max(0, p - c q)
    if (stop == k) {
      // the mass of warp w of slice r under the final residual
      auto mass = [&](int r, int w) -> float {
        if (p_ok >= 0) return ex.part[p_ok][r][w];
        if constexpr (TOPP) return reinterpret_cast<const TopPSmem *>(dyn_smem)->statp[r][w].x;
        const float4 e = ex.stat[r][w];
        return e.y > 0.f ? e.y * fast_exp2((e.x - Ml) * l2s) / Sp : 0.f;
      };
      float slice[kMaxCS];
      float total = 0.f;
      if (CS == 2 && p_ok >= 0) {
        // the last round's halves: the same sums as the loop below
#pragma unroll
        for (int r = 0; r < kMaxCS; ++r) slice[r] = r == 0 ? slice_lo : (r == 1 ? slice_hi : 0.f);
        total = (0.f + slice_lo) + slice_hi;
      } else {
#pragma unroll
        for (int r = 0; r < kMaxCS; ++r) {
          slice[r] = r < CS ? warp_sum(lane < kRWarps ? mass(r, lane) : 0.f) : 0.f;
          total += slice[r];
        }
      }
      const float target = ns.u_fb * total;
      int owner = -1;
      float prefix = 0.f, run = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxCS; ++r) {
        if (owner < 0 && r < CS && run + slice[r] > target) {
          owner = r;
          prefix = run;
        }
        run += slice[r];
      }
      if (owner < 0) {  // rounding kept the running sum below the target
        run = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCS; ++r) {
          if (r < CS && slice[r] > 0.f) {
            owner = r;
            prefix = run;
          }
          run += slice[r];
        }
        if (owner < 0) owner = 0;
      }
      writer = owner;
      // the root whose walk ends here arrives before its draw
      if (rank == owner && c.u == 0 && c.count) early = root_arrive_early(a, c, ts);
      if (rank == owner) {
        // level 1: the slice's 16 warp ranges
        const float v1 = lane < kRWarps ? mass(rank, lane) : 0.f;
        const float inc1 = warp_scan(v1, lane);
        const uint32_t hit1 = __ballot_sync(0xffffffffu, lane < kRWarps && prefix + inc1 > target);
        const int sw = hit1 ? __ffs(hit1) - 1 : -1;
        if (sw >= 0 && w_id == sw) {
          float run2 = __shfl_sync(0xffffffffu, prefix + inc1 - v1, sw);
          // level 2: the warp's eight 128-entry steps
          float ls[kRVec];
#pragma unroll
          for (int m = 0; m < kRVec; ++m) ls[m] = sum4_resid(xp[m], xq[m], c_prev);
          const float own = step_totals(ls, lane);
          float cs_all[kRVec];
#pragma unroll
          for (int m = 0; m < kRVec; ++m) cs_all[m] = __shfl_sync(0xffffffffu, own, 4 * m);
          int ms = -1;
          float before = run2;
#pragma unroll
          for (int m = 0; m < kRVec; ++m) {
            const float cs_ = cs_all[m];
            if (ms < 0 && run2 + cs_ > target) {
              ms = m;
              before = run2;
            }
            run2 += cs_;
          }
          int pick = -1;
          bool pick_near = false;
          float cb0 = target, cb1 = target;
          if (ms >= 0) {
            // level 3: the step's lanes; level 4: the lane's four entries
            float lsv = 0.f;
#pragma unroll
            for (int m = 0; m < kRVec; ++m) if (m == ms) lsv = ls[m];
            const float inc3 = warp_scan(lsv, lane);
            const uint32_t hit3 = __ballot_sync(0xffffffffu, before + inc3 > target);
            if (hit3) {
              const int L = __ffs(hit3) - 1;
              if (lane == L) {
                float4 pp = xp[0], qq = xq[0];
#pragma unroll
                for (int m = 1; m < kRVec; ++m) if (m == ms) { pp = xp[m]; qq = xq[m]; }
                float cum = before + inc3 - lsv;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                  const float wv = resid(pick4(pp, cc), pick4(qq, cc), c_prev);
                  if (pick < 0 && cum + wv > target) {
                    pick = base + 128 * ms + cc;
                    cb0 = cum;
                    cb1 = cum + wv;
                    // top-p: a drawn entry near tau (filtered values compared
                    // with tau filtered the same way)
                    pick_near = ((near & 1) && near_bits(__float_as_uint(pick4(pp, cc)), tau_kept[0])) ||
                                ((near & 2) && near_bits(__float_as_uint(pick4(qq, cc)), tau_kept[1]));
                  }
                  cum += wv;
                }
                if (pick < 0) {  // rounding: the lane's last entry of positive weight
                  for (int cc = 3; cc >= 0 && pick < 0; --cc)
                    if (resid(pick4(pp, cc), pick4(qq, cc), c_prev) > 0.f) pick = base + 128 * ms + cc;
                  if (pick < 0) pick = base + 128 * ms;
                  cb0 = cb1 = target;
                }
              }
              pick = __shfl_sync(0xffffffffu, pick, L);
              pick_near = __shfl_sync(0xffffffffu, pick_near, L);
              cb0 = __shfl_sync(0xffffffffu, cb0, L);
              cb1 = __shfl_sync(0xffffffffu, cb1, L);
            }
          }
          if (pick < 0) {
            // rounding: the warp range's last entry of positive weight
            int mine = -1;
#pragma unroll
            for (int m = 0; m < kRVec; ++m)
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                if (resid(pick4(xp[m], cc), pick4(xq[m], cc), c_prev) > 0.f) mine = base + 128 * m + cc;
            pick = __reduce_max_sync(0xffffffffu, mine);
            if (pick < 0) pick = v0 + sw * kRSpan;
            cb0 = cb1 = target;
          }
          if (lane == 0) {
            const bool tie = pick_near || fabsf(target - cb0) < kTieBand * total ||
                             fabsf(target - cb1) < kTieBand * total;
            a.fallback[t] = pick | (tie ? (1 << 31) : 0);
            ts.stop_fb = pick | (tie ? (1 << 31) : 0);
          }
        } else if (sw < 0) {
          // rounding: the slice's last entry of positive weight
          int mine = -1;
#pragma unroll
          for (int m = 0; m < kRVec; ++m)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              if (resid(pick4(xp[m], cc), pick4(xq[m], cc), c_prev) > 0.f) mine = base + 128 * m + cc;
          mine = __reduce_max_sync(0xffffffffu, mine);
          if (lane == 0) ex.last[w_id] = mine;
          __syncthreads();
          if (tid == 0) {
            int pick = -1;
            for (int w = 0; w < kRWarps; ++w) pick = max(pick, ex.last[w]);
            if (pick < 0) pick = v0;
            a.fallback[t] = pick | (1 << 31);
            ts.stop_fb = pick | (1 << 31);
          }
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
                    child_ties + ((fb >> 31) & 1), cta_timeout, !TOPP, early);
  }
  if (CS > 1) cluster_wait();
}

int launch_verify_reg(const VerifyArgs &args_in, int cs, bool top_p, cudaStream_t stream) {
  VerifyArgs args = args_in;
  args.prefetch_rows = static_cast<long long>(args.T) * cs <= sm_count() ? 1 : 0;   // one CTA per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(args.T) * cs, 1, 1);
  cfg.blockDim = dim3(kRThreads, 1, 1);
  cfg.dynamicSmemBytes = top_p ? sizeof(TopPSmem) : 0;
  if (top_p) {
    static std::atomic<size_t> granted[kMaxDevices];
    if (!allow_dynamic_smem(tree_verify_reg_kernel<true>, sizeof(TopPSmem), granted))
      return SPEC_ERR_CUDA;
  }
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attribute(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = top_p ? cudaLaunchKernelEx(&cfg, tree_verify_reg_kernel<true>, args)
                              : cudaLaunchKernelEx(&cfg, tree_verify_reg_kernel<false>, args);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace spec
