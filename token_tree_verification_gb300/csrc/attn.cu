// Steps A2 and A3: tree attention over a contiguous KV cache with a split-KV
// merge.
//
// SpecInfer developer article §2.1, tree_attention snippet: scores of the
// queries against the keys, masked entries removed, softmax, times V.
// SpecInfer news write-up, "Token 樹驗證器": the tree's K/V are appended to
// the cache depth-first so every path decodes in one pass; the mask matrix
// restricts node i to the prefix and its own ancestors.
//
// bf16 path (tree_attn_mma_kernel)
//   grid  = (splits, row blocks, B * Hkv), cluster = (splits, 1, 1)
//   CTA   = 4 consumer warps (16 query rows each: rows are (node, head in
//           group) pairs of one KV head, so one KV tile feeds all G heads)
//           + 1 producer warp that streams 64-key K and V tiles with 128B-
//           swizzled TMA tile loads into a ring of shared-memory stages.
//   math  = QK^T and PV on the tensor cores (mma.sync m16n8k16 bf16, fp32
//           accumulate), online softmax in registers in the log2 domain,
//           tree tiles masked with the node's ancestor bitmask.
//   merge = the splits of one (row block, request, KV head) form a thread
//           block cluster; their partial (m, l, O) meet in distributed shared
//           memory, so no partial result touches global memory.
// fp32 path (tree_attn_f32_kernel): one CTA per (node, head), plain FFMA, for
// fp32 inputs (small correctness workloads).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attn_common.cuh"

namespace spec {

constexpr int kMmaWarps = 4;
constexpr int kMmaRows = 16 * kMmaWarps;
constexpr int kMmaThreads = 32 * (kMmaWarps + 1);
constexpr int kMmaStages = 3;

template <int D>
struct MmaCfg {
  static constexpr int kBoxes = D / 64;                  // 128-byte SW128 boxes per key row
  static constexpr int kBoxBytes = kKeyTile * 128;       // one box: 64 keys x 64 dims bf16
  static constexpr int kTileBytes = kKeyTile * D * 2;    // K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kMergeStride = D + 8;             // floats per row of the merge buffer
  static constexpr int kSmem = kMmaStages * kStageBytes + 1024;
  static_assert(kMmaRows * kMergeStride * 4 <= kMmaStages * kStageBytes, "merge buffer");
};

__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// x, y -> bf16x2 high parts and bf16x2 remainders (x - hi, y - hi).
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = pack_bf16(x - hf.x, y - hf.y);
}

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kMmaWarps) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kMmaThreads)
tree_attn_mma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using C = MmaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMmaStages];
  __shared__ __align__(8) uint64_t empty_bar[kMmaStages];
  __shared__ float s_m[kMmaRows], s_l[kMmaRows];
  __shared__ int s_timeout;

  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_addr(smem);
  const int CS = static_cast<int>(cluster_size());
  const int split = static_cast<int>(cluster_rank());
  const int rb = blockIdx.y;
  const int b = blockIdx.z / a.Hkv;
  const int g = blockIdx.z % a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const ReqGeom R = request_geometry(a, b);
  const int rows_total = R.n * a.G;
  const int row0 = rb * kMmaRows;
  if (R.err) {
    if (tid == 0 && split == 0 && rb == 0 && g == 0) report(a.status, b, R.err);
    return;  // uniform across the cluster: same request
  }
  if (row0 >= rows_total) return;  // uniform across the cluster: same row block

  const int tiles_total = (R.keys + kKeyTile - 1) / kKeyTile;
  const int per = (tiles_total + CS - 1) / CS;
  const int t0 = split * per;
  const int ntiles = max(0, min(t0 + per, tiles_total) - t0);

  if (tid == 0) {
    for (int s = 0; s < kMmaStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kMmaWarps);
    }
    fence_barrier_init();
    s_timeout = 0;
  }
  __syncthreads();

  // per-thread state of the consumer warps
  float o[D / 8][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const int r_local[2] = {warp * 16 + (lane >> 2), warp * 16 + (lane >> 2) + 8};

  if (warp == kMmaWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kMmaStages;
        if (i >= kMmaStages && !mbar_wait(&empty_bar[st], ((i / kMmaStages) - 1) & 1)) {
          s_timeout = 1;
          break;
        }
        mbar_arrive_expect_tx(&full_bar[st], C::kStageBytes);
        const int key0 = (t0 + i) * kKeyTile;
        uint8_t *kdst = smem + st * C::kStageBytes;
        uint8_t *vdst = kdst + C::kTileBytes;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_4d(kdst + bx * C::kBoxBytes, &tmk, &full_bar[st], bx * 64, key0, g, b);
          tma_load_4d(vdst + bx * C::kBoxBytes, &tmv, &full_bar[st], bx * 64, key0, g, b);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Row -> (node, head).  Rows past the request's last row are padding.
    uint4 msk[2];
    uint32_t qa[D / 16][4];
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int r = row0 + r_local[h2];
      msk[h2] = make_uint4(0, 0, 0, 0);
      if (r < rows_total) msk[h2] = node_mask(a, R, b, R.lo + r / a.G);
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = row0 + r_local[j & 1];
        const int col = ks * 16 + 2 * (lane & 3) + ((j >> 1) << 3);
        uint32_t v = 0;
        if (r < rows_total) {
          const int node = r / a.G, head = g * a.G + r % a.G;
          if (in_bounds(R.lo + node, a.T, a.status, b))
            v = __ldg(reinterpret_cast<const uint32_t *>(
                q + (static_cast<size_t>(R.lo + node) * a.Hq + head) * D + col));
        }
        qa[ks][j] = v;
      }
    }
#pragma unroll
    for (int nb = 0; nb < D / 8; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;

    for (int i = 0; i < ntiles; ++i) {
      const int st = i % kMmaStages;
      if (!mbar_wait(&full_bar[st], (i / kMmaStages) & 1)) {
        s_timeout = 1;
        break;
      }
      const int key0 = (t0 + i) * kKeyTile;
      const uint32_t kaddr = smem_base + st * C::kStageBytes;
      const uint32_t vaddr = kaddr + C::kTileBytes;
      if (key0 + kKeyTile > R.keys) {
        // Cache slots past the request's last key may hold anything (NaN
        // included); zero those V rows so 0-weight terms stay exact zeros.
        const int valid = R.keys - key0;
        const int chunks = (kKeyTile - valid) * C::kBoxes * 8;
        uint8_t *vrow = smem + st * C::kStageBytes + C::kTileBytes;
        for (int c = tid; c < chunks; c += 32 * kMmaWarps) {
          const int row = valid + c / (C::kBoxes * 8);
          const int rest = c % (C::kBoxes * 8);
          *reinterpret_cast<uint4 *>(vrow + (rest >> 3) * C::kBoxBytes + row * 128 + (rest & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        consumer_bar();
      }
      // S = Q K^T for this warp's 16 rows and the tile's 64 keys
      float s[8][4];
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int box = ks >> 2;
        const int c16 = (ks & 3) * 2 + ((lane >> 3) & 1);
#pragma unroll
        for (int nbp = 0; nbp < 4; ++nbp) {
          const int key = nbp * 16 + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kaddr + box * C::kBoxBytes + sw128_offset(key, c16), b0, b1, b2, b3);
          mma_16816(s[2 * nbp], qa[ks], b0, b1);
          mma_16816(s[2 * nbp + 1], qa[ks], b2, b3);
        }
      }
      // scale, mask, online softmax (log2 domain)
      const bool need_mask = key0 + kKeyTile > R.L;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[nb][e] * a.scale_log2;
          if (need_mask) {
            const int key = key0 + nb * 8 + 2 * (lane & 3) + (e & 1);
            if (!key_visible(key, R.L, R.keys, msk[e >> 1])) v = -INFINITY;
          }
          s[nb][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      }
      float alpha[2], base[2], rs[2] = {0.f, 0.f};
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
        mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
        const float m_new = fmaxf(m_run[h2], mx[h2]);
        base[h2] = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[h2] = (m_run[h2] == -INFINITY) ? 0.f : exp2f(m_run[h2] - base[h2]);
        m_run[h2] = m_new;
      }
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = exp2f(s[nb][e] - base[e >> 1]);
          s[nb][e] = p;
          rs[e >> 1] += p;
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) l_run[h2] = l_run[h2] * alpha[h2] + rs[h2];
#pragma unroll
      for (int nb = 0; nb < D / 8; ++nb) {
        o[nb][0] *= alpha[0];
        o[nb][1] *= alpha[0];
        o[nb][2] *= alpha[1];
        o[nb][3] *= alpha[1];
      }
      // O += P V.  P is re-used from the S accumulators as A fragments, split
      // into a bf16 high part and a bf16 remainder so the weights keep ~16
      // significant bits: with few visible keys a single bf16 rounding of P
      // would dominate the error of small outputs.
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4], pl[4];
        split_bf16(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
        split_bf16(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
        split_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
        split_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
        const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          const int dch = np * 2 + (lane >> 4);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vaddr + (dch >> 3) * C::kBoxBytes + sw128_offset(key, dch & 7), r0, r1, r2, r3);
          mma_16816(o[2 * np], ph, r0, r1);
          mma_16816(o[2 * np + 1], ph, r2, r3);
          mma_16816(o[2 * np], pl, r0, r1);
          mma_16816(o[2 * np + 1], pl, r2, r3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
    }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 1);
      l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 2);
    }
  }
  __syncthreads();  // all stages consumed; the ring is free for the merge
  if (s_timeout && tid == 0) report(a.status, b, SPEC_ERR_TIMEOUT);

  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.o);
  if (CS == 1) {
    if (warp < kMmaWarps) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int r = row0 + r_local[h2];
        if (r >= rows_total) continue;
        const int node = r / a.G, head = g * a.G + r % a.G;
        if (!in_bounds(R.lo + node, a.T, a.status, b)) continue;
        const float inv = 1.f / l_run[h2];
        __nv_bfloat16 *dst = out + (static_cast<size_t>(R.lo + node) * a.Hq + head) * D;
#pragma unroll
        for (int nb = 0; nb < D / 8; ++nb) {
          *reinterpret_cast<uint32_t *>(dst + nb * 8 + 2 * (lane & 3)) =
              pack_bf16(o[nb][2 * h2] * inv, o[nb][2 * h2 + 1] * inv);
        }
      }
    }
    return;
  }

  // ---- split merge through distributed shared memory
  float *obuf = reinterpret_cast<float *>(smem);
  if (warp < kMmaWarps) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float *row = obuf + r_local[h2] * C::kMergeStride;
#pragma unroll
      for (int nb = 0; nb < D / 8; ++nb)
        *reinterpret_cast<float2 *>(row + nb * 8 + 2 * (lane & 3)) =
            make_float2(o[nb][2 * h2], o[nb][2 * h2 + 1]);
      if ((lane & 3) == 0) {
        s_m[r_local[h2]] = m_run[h2];
        s_l[r_local[h2]] = l_run[h2];
      }
    }
  }
  cluster_sync_all();
  const int rpr = kMmaRows / CS;
  const int nvec = rpr * (D / 4);
  for (int idx = tid; idx < nvec; idx += kMmaThreads) {
    const int lr = split * rpr + idx / (D / 4);
    const int c4 = idx % (D / 4);
    const int r = row0 + lr;
    if (r >= rows_total) continue;
    float M = -INFINITY;
    for (int s2 = 0; s2 < CS; ++s2) M = fmaxf(M, ld_peer_f32(peer_addr(&s_m[lr], s2)));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    for (int s2 = 0; s2 < CS; ++s2) {
      const float ms = ld_peer_f32(peer_addr(&s_m[lr], s2));
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - M);
      L += w * ld_peer_f32(peer_addr(&s_l[lr], s2));
      const float4 v = ld_peer_f32x4(peer_addr(obuf + lr * C::kMergeStride + c4 * 4, s2));
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    const float inv = 1.f / L;
    const int node = r / a.G, head = g * a.G + r % a.G;
    if (!in_bounds(R.lo + node, a.T, a.status, b)) continue;
    __nv_bfloat16 *dst = out + (static_cast<size_t>(R.lo + node) * a.Hq + head) * D + c4 * 4;
    uint2 pk;
    pk.x = pack_bf16(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(dst) = pk;
  }
  cluster_sync_all();  // peers may still be reading this CTA's buffers
}

// ---------------------------------------------------------------- fp32 path
constexpr int kF32Threads = 128;
constexpr int kF32Chunk = 128;  // keys scored per round

__global__ void __launch_bounds__(kF32Threads)
tree_attn_f32_kernel(const AttnArgs a) {
  __shared__ float qs[128];
  __shared__ float ps[kF32Chunk];
  __shared__ float red[kF32Threads / 32];
  const int h = blockIdx.x, t = blockIdx.y, tid = threadIdx.x;
  const int D = a.D;
  const int b = find_request(a.offsets, a.B, t);
  if (b < 0) return;
  const ReqGeom R = request_geometry(a, b);
  if (R.err) {
    if (tid == 0 && h == 0 && t == R.lo) report(a.status, b, R.err);
    return;
  }
  const int g = h / a.G;
  const uint4 m = node_mask(a, R, b, t);
  const float *q = static_cast<const float *>(a.q) + (static_cast<size_t>(t) * a.Hq + h) * D;
  const size_t kv_off = (static_cast<size_t>(b) * a.Hkv + g) * a.S_cap * D;
  const float *kc = static_cast<const float *>(a.k) + kv_off;
  const float *vc = static_cast<const float *>(a.v) + kv_off;
  if (tid < D) qs[tid] = q[tid];
  __syncthreads();
  float m_run = -INFINITY, l_run = 0.f, acc = 0.f;
  for (int c0 = 0; c0 < R.keys; c0 += kF32Chunk) {
    // scores of this chunk, one key per thread (log2 domain)
    const int key = c0 + tid;
    float sc = -INFINITY;
    if (key < R.keys && key_visible(key, R.L, R.keys, m) && in_bounds(key, a.S_cap, a.status, b)) {
      const float *kr = kc + static_cast<size_t>(key) * D;
      float dot = 0.f;
      for (int d = 0; d < D; ++d) dot = fmaf(qs[d], kr[d], dot);
      sc = dot * a.scale_log2;
    }
    float mx = sc;
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < kF32Threads / 32; ++w) mx = fmaxf(mx, red[w]);
    const float m_new = fmaxf(m_run, mx);
    const float base = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - base);
    const float p = exp2f(sc - base);
    ps[tid] = p;
    float sum = p;
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = sum;
    __syncthreads();
    sum = 0.f;
    for (int w = 0; w < kF32Threads / 32; ++w) sum += red[w];
    l_run = l_run * alpha + sum;
    m_run = m_new;
    // weighted values, one output dimension per thread
    if (tid < D) {
      float part = 0.f;
      const int nk = min(kF32Chunk, R.keys - c0);
      for (int j = 0; j < nk; ++j)
        if (ps[j] != 0.f && in_bounds(c0 + j, a.S_cap, a.status, b))
          part = fmaf(ps[j], vc[static_cast<size_t>(c0 + j) * D + tid], part);
      acc = acc * alpha + part;
    }
    __syncthreads();
  }
  if (tid < D) static_cast<float *>(a.o)[(static_cast<size_t>(t) * a.Hq + h) * D + tid] = acc / l_run;
}

}  // namespace spec

// ---------------------------------------------------------------- host side
namespace {

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn tensor_map_encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// 4-D map over a [B][Hkv][S_cap][D] bf16 cache; one box is 64 keys x 64 dims
// (128 bytes per key row), loaded with 128-byte swizzle.  Reads past S_cap
// are zero-filled by the hardware.
bool encode_kv_map(CUtensorMap *m, const void *base, int B, int Hkv, int S_cap, int D) {
  EncodeFn enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S_cap),
                        static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(S_cap) * D * 2,
                           static_cast<cuuint64_t>(Hkv) * S_cap * D * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(spec::kKeyTile), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over q [T][Hq][D] bf16 whose box is one query block of a KV head:
// 64 dims x G heads x (rows / G) nodes, loaded with 128-byte swizzle so the
// block lands as `rows` rows of 128 bytes (node-major, head-minor).
bool encode_q_map(CUtensorMap *m, const void *base, int T, int Hq, int G, int D, int rows) {
  EncodeFn enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(rows / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Which bf16 kernel runs: tcgen05 by default; SPEC_TREE_ATTN_KERNEL=mma
// selects the mma.sync kernel (kept as a second implementation for testing).
bool use_mma_kernel() {
  const char *e = getenv("SPEC_TREE_ATTN_KERNEL");
  return e != nullptr && strcmp(e, "mma") == 0;
}

template <int D>
int launch_mma(const spec::AttnArgs &args, int max_prefix, int T, cudaStream_t stream) {
  using C = spec::MmaCfg<D>;
  auto kernel = spec::tree_attn_mma_kernel<D>;
  static std::atomic<size_t> granted[spec::kMaxDevices];
  if (!spec::allow_dynamic_smem(kernel, C::kSmem, granted)) return SPEC_ERR_CUDA;
  static std::atomic<int> occupancy[spec::kMaxDevices];   // resident CTAs per SM, per device
  const int dev = spec::current_device();
  int per_sm = dev >= 0 ? occupancy[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm < 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, spec::kMmaThreads, C::kSmem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    if (dev >= 0) occupancy[dev].store(per_sm, std::memory_order_relaxed);
  }
  CUtensorMap tmk, tmv;
  if (!encode_kv_map(&tmk, args.k, args.B, args.Hkv, args.S_cap, D) ||
      !encode_kv_map(&tmv, args.v, args.B, args.Hkv, args.S_cap, D))
    return SPEC_ERR_CUDA;
  const int max_nodes = T < SPEC_MAX_TREE_NODES ? T : SPEC_MAX_TREE_NODES;
  const int rowblocks = (max_nodes * args.G + spec::kMmaRows - 1) / spec::kMmaRows;
  const long long max_keys = static_cast<long long>(max_prefix) + max_nodes;
  const int tiles_max = static_cast<int>((max_keys + spec::kKeyTile - 1) / spec::kKeyTile);
  const long long units = static_cast<long long>(rowblocks) * args.B * args.Hkv;
  const long long slots = static_cast<long long>(per_sm) * spec::sm_count();
  // splits: enough that no CTA streams more than ~16 tiles, then more while
  // the grid still fits in one wave
  int cs = 1;
  while (cs < 8 && tiles_max > 16 * cs) cs *= 2;
  while (cs < 8 && units * cs * 2 <= slots && tiles_max >= 2 * cs) cs *= 2;
  if (units > 65535) return SPEC_ERR_SHAPE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, rowblocks, static_cast<unsigned>(args.B * args.Hkv));
  cfg.blockDim = dim3(spec::kMmaThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args, tmk, tmv) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" size_t spec_tree_attn_workspace_size(int B, int T, int Hq, int Hkv, int D,
                                                int max_prefix) {
  (void)B; (void)T; (void)Hq; (void)Hkv; (void)D; (void)max_prefix;
  return 0;  // key splits merge on chip, within a thread-block cluster
}

extern "C" int spec_tree_attn(const void *q, const void *k_cache, const void *v_cache, void *o,
                              int dtype, int B, int T, int Hq, int Hkv, int D, int S_cap,
                              int max_prefix, const int32_t *prefix_lens,
                              const int32_t *tree_offsets, const uint32_t *mask,
                              float softmax_scale, void *workspace, size_t workspace_bytes,
                              int32_t *status, void *stream) {
  return spec_tree_attn_ex(q, k_cache, v_cache, o, dtype, B, T, Hq, Hkv, D, S_cap, max_prefix,
                           prefix_lens, tree_offsets, mask, nullptr, softmax_scale, workspace,
                           workspace_bytes, 0, status, stream);
}

extern "C" int spec_tree_attn_ex(const void *q, const void *k_cache, const void *v_cache, void *o,
                                 int dtype, int B, int T, int Hq, int Hkv, int D, int S_cap,
                                 int max_prefix, const int32_t *prefix_lens,
                                 const int32_t *tree_offsets, const uint32_t *mask,
                                 const int32_t *parents, float softmax_scale, void *workspace,
                                 size_t workspace_bytes, int max_ctas, int32_t *status,
                                 void *stream) {
  if (max_ctas < 0) return SPEC_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !o || !prefix_lens || !tree_offsets || (!mask && !parents) ||
      !status)
    return SPEC_ERR_NULL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 1 || T < 1 || T > B * SPEC_MAX_TREE_NODES || Hq < 1 || Hkv < 1 || Hq % Hkv ||
      S_cap < 1 || max_prefix < 0)
    return SPEC_ERR_SHAPE;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return SPEC_ERR_SHAPE;
  if (D != 64 && D != 128) return SPEC_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(o) |
       reinterpret_cast<uintptr_t>(mask)) & 15)
    return SPEC_ERR_ALIGNMENT;
  spec::AttnArgs args;
  args.q = q;
  args.k = k_cache;
  args.v = v_cache;
  args.o = o;
  args.prefix_lens = prefix_lens;
  args.offsets = tree_offsets;
  args.mask = reinterpret_cast<const uint4 *>(mask);
  args.parents = mask ? nullptr : parents;
  args.status = status;
  args.B = B;
  args.T = T;
  args.Hq = Hq;
  args.Hkv = Hkv;
  args.G = G;
  args.D = D;
  args.S_cap = S_cap;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(D));
  args.scale_log2 = scale * 1.4426950408889634f;
  args.rows_per_cta = spec::kMmaRows;
  // a single request holds T nodes; with max_prefix exact its key count is known
  args.prefetch_keys = B == 1 ? max_prefix + T : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SPEC_F32) {
    spec::tree_attn_f32_kernel<<<dim3(Hq, T), spec::kF32Threads, 0, st>>>(args);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  if (use_mma_kernel())
    return D == 128 ? launch_mma<128>(args, max_prefix, T, st) : launch_mma<64>(args, max_prefix, T, st);
  // every row block holds at most 64 rows: the packed tcgen05 variant
  const bool packed = (T < SPEC_MAX_TREE_NODES ? T : SPEC_MAX_TREE_NODES) * G <= 64;
  CUtensorMap tmq, tmk, tmv;
  if (!encode_q_map(&tmq, q, T, Hq, G, D, packed ? 64 : 128) ||
      !encode_kv_map(&tmk, k_cache, B, Hkv, S_cap, D) ||
      !encode_kv_map(&tmv, v_cache, B, Hkv, S_cap, D))
    return SPEC_ERR_CUDA;
  (void)workspace; (void)workspace_bytes;
  // the key splits are planned for the SMs the caller leaves to this launch
  const int sms = spec::sm_count();
  return spec::launch_attn_tc(args, max_prefix, T, tmq, tmk, tmv, packed,
                              max_ctas > 0 && max_ctas < sms ? max_ctas : sms, st);
}
