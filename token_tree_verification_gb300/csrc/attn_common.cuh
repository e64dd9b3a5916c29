// Shared pieces of the tree-attention kernels: argument block, per-request
// key geometry, visibility of a key to a row, and the SW128 smem addressing
// produced by TMA tile loads.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace spec {

constexpr int kKeyTile = 64;   // keys per TMA tile

struct AttnArgs {
  const void *q;
  const void *k;           // [B][Hkv][S_cap][D] (read directly by the fp32 path)
  const void *v;
  void *o;
  const int32_t *prefix_lens;
  const int32_t *offsets;
  const uint4 *mask;       // per node ancestor-or-self bits, or null: built from `parents`
  const int32_t *parents;  // [T] request-local parent of every node (read when mask is null)
  int32_t *status;
  int B, T, Hq, Hkv, G, D, S_cap;
  float scale_log2;        // softmax scale * log2(e)
  int rows_per_cta;        // rows of one CTA (node-major, head-minor)
  int prefetch_keys;       // > 0: the key count the host expects for a single request
                           // (its L2 prefetch of the first tiles may start early)
};

// Geometry of request b as one CTA sees it.  Keys [0, L) are the prefix,
// keys [L, L + n) the tree slots in node order.
struct ReqGeom {
  int lo, n, L, keys, err;
};

__device__ __forceinline__ ReqGeom request_geometry(const AttnArgs &a, int b) {
  ReqGeom r;
  r.lo = __ldg(a.offsets + b);
  const int hi = __ldg(a.offsets + b + 1);
  r.n = hi - r.lo;
  r.L = __ldg(a.prefix_lens + b);
  r.err = 0;
  if (r.lo < 0 || hi > a.T || r.n < 1 || r.n > SPEC_MAX_TREE_NODES) r.err = SPEC_ERR_TREE_TOO_LARGE;
  else if (r.L < 0 || r.L + r.n > a.S_cap) r.err = SPEC_ERR_PREFIX_RANGE;
  r.keys = r.err ? 0 : r.L + r.n;
  return r;
}

// Key `key` is visible to a row whose node has ancestor set `m` (bits >= n
// already cleared): prefix keys always, tree key L + a iff bit a is set.
__device__ __forceinline__ bool key_visible(int key, int L, int keys, const uint4 &m) {
  if (key < L) return true;
  if (key >= keys) return false;
  const int a = key - L;
  const uint32_t w = (a < 64) ? ((a < 32) ? m.x : m.y) : ((a < 96) ? m.z : m.w);
  return (w >> (a & 31)) & 1u;
}

// Ancestor set of a node with bits at or above n cleared, so a malformed mask
// can never make the kernels read tree slots the request does not own.
__device__ __forceinline__ uint4 clip_mask(uint4 m, int n) {
  uint32_t *w = &m.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int lo = 32 * i;
    if (n <= lo) w[i] = 0;
    else if (n < lo + 32) w[i] &= (1u << (n - lo)) - 1u;
  }
  return m;
}

// Ancestor-or-self set of request-local node u (u < n <= 128), from the
// request's parent array read through par(i): the walk follows u's parent
// chain to the root.  Every step must go to a lower index and end at a root
// whose parent is -1; a parent that breaks this ends the walk (so a malformed
// array can never loop) and sets *bad.
template <typename Par>
__device__ __forceinline__ uint4 ancestor_mask(Par par, int u, bool *bad) {
  uint4 m = make_uint4(0u, 0u, 0u, 0u);
  int x = u;
  for (;;) {
    const uint32_t bit = 1u << (x & 31);
    const int q = x >> 5;
    m.x |= q == 0 ? bit : 0u;
    m.y |= q == 1 ? bit : 0u;
    m.z |= q == 2 ? bit : 0u;
    m.w |= q == 3 ? bit : 0u;
    const int p = par(x);
    if (x == 0) {
      if (p != -1) *bad = true;
      break;
    }
    if (p < 0 || p >= x) {
      *bad = true;
      break;
    }
    x = p;
  }
  return m;
}

// The mask of row node t (global index) of request R, for the kernels that
// do not stage the parent array: from the mask array when there is one,
// else by walking the parents in global memory.  A malformed parent array
// reports SPEC_ERR_BAD_PARENT for the request.
// (the walk is kept out of line, so that the kernels' mask-array path is
// compiled as without it)
static __device__ __noinline__ uint4 node_mask_walk(const AttnArgs &a, const ReqGeom &R, int b, int t) {
  bool bad = false;
  const int32_t *par = a.parents + R.lo;
  const uint4 m = ancestor_mask(
      [&](int i) { return in_bounds(R.lo + i, a.T, a.status, b) ? __ldg(par + i) : -2; }, t - R.lo,
      &bad);
  if (bad) report(a.status, b, SPEC_ERR_BAD_PARENT);
  return m;
}

__device__ __forceinline__ uint4 node_mask(const AttnArgs &a, const ReqGeom &R, int b, int t) {
  if (a.mask) {
    if (!in_bounds(t, a.T, a.status, b)) return make_uint4(0u, 0u, 0u, 0u);
    return clip_mask(__ldg(a.mask + t), R.n);
  }
  return node_mask_walk(a, R, b, t);
}

// Byte offset of 16-byte chunk `c16` (0..7) of row `row` inside one SW128
// box of 128-byte rows (the layout a 128B-swizzled TMA load writes when the
// box starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t sw128_offset(int row, int c16) {
  return static_cast<uint32_t>(row * 128 + ((c16 ^ (row & 7)) << 4));
}

// tcgen05 path (attn_tc.cu).  `packed`: every row block has at most 64 rows
// (the Q map's box then holds 64 rows).
int launch_attn_tc(const AttnArgs &args, int max_prefix, int T, const CUtensorMap &tmq,
                   const CUtensorMap &tmk, const CUtensorMap &tmv, bool packed, int num_sms,
                   cudaStream_t stream);

}  // namespace spec
