// Steps A2 and A3 on the 5th-generation tensor cores (tcgen05), bf16 in,
// fp32 accumulate.
//
// SpecInfer developer article §2.1, tree_attention snippet (masked scores,
// softmax, times V); SpecInfer news write-up "Token 樹驗證器" (tree K/V
// appended to the cache depth-first, mask restricted to the node's ancestors).
//
// One CTA = one key split x one block of 128 query rows x one (request, KV
// head).  Rows are (node, head-in-group) pairs, so one K/V tile feeds all G
// query heads of the KV head.  Warp roles:
//   warp 0      TMA producer: the Q block once, then 64-key K and V tiles
//               (128-byte swizzle) into a 3-stage ring.
//   warp 1      allocates TMEM; one thread issues the MMAs:
//                 S_i = Q K_i^T            M=128, N=64, K=D   (TMEM S[i%2])
//                 O  += P_i V_i (hi, lo)   M=128, N=D,  K=64  (TMEM O)
//               with S_{i+1} issued before P_i is ready, so the softmax of
//               one tile overlaps the QK^T of the next.
//   warps 2-9   two threads per TMEM lane (= query row), one per half of
//               the tile's keys: read S from TMEM, mask with the node's
//               ancestor bits, share the row max with the partner thread,
//               online softmax with a lazily moved reference max (the stored
//               O is rescaled only when a row's max grows by more than 2^8),
//               write P as bf16 high and remainder parts to shared memory.
//               With at most 64 rows the remainder part goes to the unused
//               rows 64-127 of the same P operand (one 4-MMA P V pass; the
//               two halves are added from TMEM lanes r and r + 64 at the end,
//               and the warps of lanes 64-127 mirror their rows' rescaling).
//   epilogue    the O rows leave TMEM; the splits of one cluster push their
//               (m, l, O) rows into the owning CTA's shared memory with
//               remote stores, which then merges them locally.
#include <cuda.h>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "tcgen05.cuh"

namespace spec {

constexpr int kTcRows = 128;
constexpr int kTcStages = 3;
constexpr int kTcSoftmaxWarps = 8;   // two warps (key halves) per TMEM lane quadrant
constexpr int kTcThreads = 32 * (2 + kTcSoftmaxWarps);
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct TcCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kQBoxBytes = kTcRows * 128;
  static constexpr int kQBytes = kTcRows * D * 2;
  static constexpr int kKVBoxBytes = kKeyTile * 128;
  static constexpr int kTileBytes = kKeyTile * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kPBytes = kTcRows * kKeyTile * 2;   // one of the hi / lo parts
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffP = kOffKV + kTcStages * kStageBytes;
  static constexpr int kSmem = kOffP + 2 * 2 * kPBytes + 1024;
  static constexpr int kMergeStride = D + 4;             // floats per (split, row) slot
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 128;
  // owner-side merge slots: (split, row) pairs, at most rows + 7 of them
  static_assert((kTcRows + 7) * kMergeStride * 4 <= kTcStages * kStageBytes,
                "merge buffer must fit in the K/V ring");
  static_assert(kTcRows / 2 * D * 4 <= 2 * 2 * kPBytes, "packed remainder exchange fits the P buffers");
};

__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<const uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
tree_attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kTcStages], bar_empty[kTcStages];
  __shared__ __align__(8) uint64_t bar_q, bar_s[2], bar_p[2], bar_o[2];
  __shared__ uint32_t s_tmem;
  __shared__ float x_max[2][2][kTcRows];   // [tile parity][key half][row]
  __shared__ float x_l[2][kTcRows];
  __shared__ float m_slot[8][kTcRows], l_slot[8][kTcRows];   // owner-side merge (split, row)
  __shared__ int s_timeout;

  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const int CS = static_cast<int>(cluster_size());
  const int split = static_cast<int>(cluster_rank());
  const int rb = blockIdx.y;
  const int b = blockIdx.z / a.Hkv;
  const int g = blockIdx.z % a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const ReqGeom R = request_geometry(a, b);
  const int rows_total = R.n * a.G;
  const int row0 = rb * kTcRows;
  if (R.err) {
    if (tid == 0 && split == 0 && rb == 0 && g == 0) report(a.status, b, R.err);
    return;  // uniform across the cluster
  }
  if (row0 >= rows_total) return;  // uniform across the cluster
  const int rows_here = min(kTcRows, rows_total - row0);
  // Packed mode (at most 64 rows): the bf16 remainder of P goes to rows
  // 64-127 of the same P operand, so one 4-MMA pass computes both halves
  // of P V into TMEM lanes r and r + 64.
  const bool packed = rows_here <= kTcRows / 2;
  const int tiles_total = (R.keys + kKeyTile - 1) / kKeyTile;
  const int per = (tiles_total + CS - 1) / CS;
  const int t0 = split * per;
  const int ntiles = max(0, min(t0 + per, tiles_total) - t0);
  const int rpr = (rows_here + CS - 1) / CS;   // rows merged by each CTA of the cluster

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_q, 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&bar_s[j], 1);
      mbar_init(&bar_p[j], kTcSoftmaxWarps);
      mbar_init(&bar_o[j], 1);
    }
    fence_barrier_init();
    s_timeout = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(&s_tmem, C::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  // softmax-thread geometry (warps 2..9): TMEM lane r, key / column half
  const int quad = warp & 3;
  const int half = (warp - 2) >> 2;
  const int r = quad * 32 + lane;
  // the score row this thread follows: its own, or (helper lanes 64-127 in
  // packed mode) the row whose remainder part it accumulates
  const bool helper = packed && quad >= 2;
  const int srow = helper ? r - kTcRows / 2 : r;
  const bool row_ok = srow < rows_here;
  const bool computes = warp >= 2 && !helper && quad * 32 < rows_here;   // reads S, writes P
  const bool lanes_live = warp >= 2 && (quad & (packed ? 1 : 3)) * 32 < rows_here;
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  float o_keep[D / 2];
  float m_used = -INFINITY, l_half = 0.f, l_row = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      mbar_arrive_expect_tx(&bar_q, C::kQBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx)
        tma_load_3d(smem + C::kOffQ + bx * C::kQBoxBytes, &tmq, &bar_q, bx * 64, g * a.G,
                    R.lo + row0 / a.G);
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kTcStages;
        if (i >= kTcStages && !mbar_wait(&bar_empty[st], ((i / kTcStages) - 1) & 1)) {
          s_timeout = 1;
          break;
        }
        mbar_arrive_expect_tx(&bar_full[st], C::kStageBytes);
        const int key0 = (t0 + i) * kKeyTile;
        uint8_t *kdst = smem + C::kOffKV + st * C::kStageBytes;
        uint8_t *vdst = kdst + C::kTileBytes;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_4d(kdst + bx * C::kKVBoxBytes, &tmk, &bar_full[st], bx * 64, key0, g, b);
          tma_load_4d(vdst + bx * C::kKVBoxBytes, &tmv, &bar_full[st], bx * 64, key0, g, b);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcRows, kKeyTile, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kTcRows, D, 0, 1);
      const int parts = packed ? 1 : 2;
      bool ok = mbar_wait(&bar_q, 0);
      tc::fence_after_sync();
      for (int i = 0; ok && i <= ntiles; ++i) {
        if (i < ntiles) {
          const int st = i % kTcStages;
          if (!mbar_wait(&bar_full[st], (i / kTcStages) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t kb = sb + C::kOffKV + st * C::kStageBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t ad = tc::smem_desc_sw128(
                sb + C::kOffQ + (ks >> 2) * C::kQBoxBytes + (ks & 3) * 32, 16, 1024);
            const uint64_t bd =
                tc::smem_desc_sw128(kb + (ks >> 2) * C::kKVBoxBytes + (ks & 3) * 32, 16, 1024);
            tc::mma_bf16(tmem + C::kColS + (i & 1) * kKeyTile, ad, bd, idS, ks > 0);
          }
          tc::commit(&bar_s[i & 1]);
        }
        if (i >= 1) {
          const int j = i - 1, st = j % kTcStages;
          if (!mbar_wait(&bar_p[j & 1], (j >> 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t vb = sb + C::kOffKV + st * C::kStageBytes + C::kTileBytes;
          const uint32_t pb = sb + C::kOffP + (j & 1) * 2 * C::kPBytes;
          for (int part = 0; part < parts; ++part) {
#pragma unroll
            for (int kk = 0; kk < kKeyTile / 16; ++kk) {
              const uint64_t ad = tc::smem_desc_sw128(pb + part * C::kPBytes + kk * 32, 16, 1024);
              const uint64_t bd = tc::smem_desc_sw128(vb + kk * 16 * 128, C::kKVBoxBytes, 1024);
              tc::mma_bf16(tmem + C::kColO, ad, bd, idO, (j | part | kk) != 0);
            }
          }
          tc::commit(&bar_o[j & 1]);
          tc::commit(&bar_empty[st]);
        }
      }
      if (!ok) s_timeout = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    uint4 msk = make_uint4(0, 0, 0, 0);
    if (computes && row_ok) msk = clip_mask(__ldg(a.mask + R.lo + (row0 + r) / a.G), R.n);
    const float sl2 = a.scale_log2;
    bool ok = true;
    // A timed-out wait clears `ok` and later waits are skipped, but the loop
    // runs to the end so every softmax warp meets every named barrier.
    for (int i = 0; i < ntiles; ++i) {
      if (ok && !mbar_wait(&bar_s[i & 1], (i >> 1) & 1)) ok = false;
      __syncwarp();
      tc::fence_after_sync();
      const int key0 = (t0 + i) * kKeyTile;
      const int st = i % kTcStages;
      if (key0 + kKeyTile > R.keys) {
        // V rows past the request's last key may hold anything: zero them so
        // their zero weights contribute exact zeros.
        const int valid = R.keys - key0;
        const int chunks = (kKeyTile - valid) * C::kBoxes * 8;
        uint8_t *vrow = smem + C::kOffKV + st * C::kStageBytes + C::kTileBytes;
        for (int c = tid - 64; c < chunks; c += 32 * kTcSoftmaxWarps) {
          const int row = valid + c / (C::kBoxes * 8);
          const int rest = c % (C::kBoxes * 8);
          *reinterpret_cast<uint4 *>(vrow + (rest >> 3) * C::kKVBoxBytes + row * 128 +
                                     (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      float s[32];
      bool want = false;
      if (computes) {
        tc::ld32(trow + C::kColS + (i & 1) * kKeyTile + 32 * half, s);
        tc::wait_ld();
        const int kbase = key0 + 32 * half;
        if (kbase + 32 > R.L) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (!key_visible(kbase + j, R.L, R.keys, msk)) s[j] = -INFINITY;
        }
        float mt = s[0];
#pragma unroll
        for (int j = 1; j < 32; ++j) mt = fmaxf(mt, s[j]);
        x_max[i & 1][half][r] = mt;
        want = row_ok && (mt * sl2 > m_used + kRescaleLog2);
      }
      // one barrier: both halves' maxima are visible, and whether any row of
      // the block moves its reference max
      const bool any_resc = named_bar_or(2, 32 * kTcSoftmaxWarps, want);
      const float mt = (lanes_live && row_ok)
                           ? fmaxf(x_max[i & 1][0][srow], x_max[i & 1][1][srow]) * sl2
                           : -INFINITY;
      const bool resc = row_ok && lanes_live && (mt > m_used + kRescaleLog2);
      if (any_resc) {
        const float m_new = resc ? mt : m_used;
        const float alpha = !resc ? 1.f : (m_used == -INFINITY ? 0.f : exp2f(m_used - m_new));
        if (i > 0 && lanes_live) {
          // O holds the products of tiles < i: wait for the last of them,
          // then rescale this thread's half of its TMEM lane in place.
          if (ok && !mbar_wait(&bar_o[(i - 1) & 1], ((i - 1) >> 1) & 1)) ok = false;
          __syncwarp();
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            float o[32];
            tc::ld32(trow + C::kColO + half * (D / 2) + c * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tc::st32(trow + C::kColO + half * (D / 2) + c * 32, o);
          }
          tc::wait_st();
        }
        l_half *= alpha;
        m_used = m_new;
      }
      if (computes) {
        // the P buffer of this parity is free once the P V of tile i-2 is done
        if (ok && i >= 2 && !mbar_wait(&bar_o[i & 1], ((i - 2) >> 1) & 1)) ok = false;
        __syncwarp();
        const float nbase = (m_used == -INFINITY) ? 0.f : -m_used;
        uint8_t *pbuf = smem + C::kOffP + (i & 1) * 2 * C::kPBytes;
        uint8_t *prow_hi = pbuf + r * 128;
        uint8_t *prow_lo = packed ? pbuf + (r + kTcRows / 2) * 128 : pbuf + C::kPBytes + r * 128;
        float psum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = fast_exp2(fmaf(s[cc * 8 + 2 * e], sl2, nbase));
            const float p1 = fast_exp2(fmaf(s[cc * 8 + 2 * e + 1], sl2, nbase));
            psum += p0 + p1;
            const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
            const float2 hf = __bfloat1622float2(h);
            hi[e] = bf16x2_bits(h);
            lo[e] = bf16x2_bits(__floats2bfloat162_rn(p0 - hf.x, p1 - hf.y));
          }
          const int off = ((4 * half + cc) ^ (r & 7)) << 4;   // (r + 64) & 7 == r & 7
          *reinterpret_cast<uint4 *>(prow_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4 *>(prow_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        l_half += psum;
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[i & 1]);
    }
    if (!ok) s_timeout = 1;
    // ---- epilogue: O rows out of TMEM.  Every softmax warp waits for the
    //      last P V before any thread reuses the K/V ring or P buffers.
    if (ntiles > 0) {
      if (ok && !mbar_wait(&bar_o[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) s_timeout = 1;
      __syncwarp();
      tc::fence_after_sync();
    }
#pragma unroll
    for (int e = 0; e < D / 2; ++e) o_keep[e] = 0.f;
    if (lanes_live && ntiles > 0) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        float o[32];
        tc::ld32(trow + C::kColO + half * (D / 2) + c * 32, o);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o_keep[c * 32 + e] = o[e];
      }
    }
    // packed: lanes r + 64 hold the remainder part of row r's P V
    float *xo = reinterpret_cast<float *>(smem + C::kOffP);   // [64 rows][D], P buffers are free
    if (packed && helper && row_ok) {
#pragma unroll
      for (int e = 0; e < D / 2; e += 4)
        *reinterpret_cast<float4 *>(xo + srow * D + half * (D / 2) + e) =
            make_float4(o_keep[e], o_keep[e + 1], o_keep[e + 2], o_keep[e + 3]);
    }
    if (!helper) x_l[half][r] = l_half;
    named_bar_sync(2, 32 * kTcSoftmaxWarps);
    if (!helper) {
      l_row = l_half + x_l[half ^ 1][r];
      if (packed && row_ok) {
#pragma unroll
        for (int e = 0; e < D / 2; e += 4) {
          const float4 v = *reinterpret_cast<const float4 *>(xo + r * D + half * (D / 2) + e);
          o_keep[e] += v.x;
          o_keep[e + 1] += v.y;
          o_keep[e + 2] += v.z;
          o_keep[e + 3] += v.w;
        }
      }
    }
    if (CS == 1 && !helper && row_ok && ntiles > 0) {
      const float inv = 1.f / l_row;
      const int rr = row0 + r;
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.o) +
                           (static_cast<size_t>(R.lo + rr / a.G) * a.Hq + g * a.G + rr % a.G) * D +
                           half * (D / 2);
#pragma unroll
      for (int q8 = 0; q8 < D / 16; ++q8) {
        uint4 pk;
        pk.x = bf16x2_bits(__floats2bfloat162_rn(o_keep[q8 * 8 + 0] * inv, o_keep[q8 * 8 + 1] * inv));
        pk.y = bf16x2_bits(__floats2bfloat162_rn(o_keep[q8 * 8 + 2] * inv, o_keep[q8 * 8 + 3] * inv));
        pk.z = bf16x2_bits(__floats2bfloat162_rn(o_keep[q8 * 8 + 4] * inv, o_keep[q8 * 8 + 5] * inv));
        pk.w = bf16x2_bits(__floats2bfloat162_rn(o_keep[q8 * 8 + 6] * inv, o_keep[q8 * 8 + 7] * inv));
        *reinterpret_cast<uint4 *>(dst + q8 * 8) = pk;
      }
    }
  }

  __syncwarp();
  tc::fence_before_sync();
  if (CS > 1) {
    // ---- split merge: every CTA pushes its rows into the owner's smem
    cluster_sync_all();  // every CTA of the cluster is done with its K/V ring
    if (warp >= 2 && !helper && row_ok) {
      const int owner = r / rpr;
      const int slot = split * rpr + (r - owner * rpr);
      float *mbase = reinterpret_cast<float *>(smem + C::kOffKV) + slot * C::kMergeStride + half * (D / 2);
      const uint32_t dst = peer_addr(mbase, owner);
#pragma unroll
      for (int e = 0; e < D / 2; e += 4)
        st_peer_f32x4(dst + e * 4, make_float4(o_keep[e], o_keep[e + 1], o_keep[e + 2], o_keep[e + 3]));
      if (half == 0) {
        st_peer_f32(peer_addr(&m_slot[split][r - owner * rpr], owner), ntiles > 0 ? m_used : -INFINITY);
        st_peer_f32(peer_addr(&l_slot[split][r - owner * rpr], owner), l_row);
      }
    }
    cluster_sync_all();  // the pushes have landed
    const int r_begin = split * rpr, r_end = min(rows_here, r_begin + rpr);
    const int nvec = max(0, r_end - r_begin) * (D / 4);
    const float *mb = reinterpret_cast<const float *>(smem + C::kOffKV);
    for (int idx = tid; idx < nvec; idx += kTcThreads) {
      const int lr = idx / (D / 4);
      const int c4 = idx % (D / 4);
      float M = -INFINITY;
      for (int s2 = 0; s2 < CS; ++s2) M = fmaxf(M, m_slot[s2][lr]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float L = 0.f;
      for (int s2 = 0; s2 < CS; ++s2) {
        const float ms = m_slot[s2][lr];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        L += w * l_slot[s2][lr];
        const float4 v = *reinterpret_cast<const float4 *>(mb + (s2 * rpr + lr) * C::kMergeStride + c4 * 4);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
      const float inv = 1.f / L;
      const int rr = row0 + r_begin + lr;
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.o) +
                           (static_cast<size_t>(R.lo + rr / a.G) * a.Hq + g * a.G + rr % a.G) * D + c4 * 4;
      uint2 pk;
      pk.x = bf16x2_bits(__floats2bfloat162_rn(acc.x * inv, acc.y * inv));
      pk.y = bf16x2_bits(__floats2bfloat162_rn(acc.z * inv, acc.w * inv));
      *reinterpret_cast<uint2 *>(dst) = pk;
    }
  }
  __syncthreads();
  tc::fence_after_sync();
  if (s_timeout && tid == 0) report(a.status, b, SPEC_ERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

template __global__ void tree_attn_tc_kernel<64>(const AttnArgs, const __grid_constant__ CUtensorMap,
                                                 const __grid_constant__ CUtensorMap,
                                                 const __grid_constant__ CUtensorMap);
template __global__ void tree_attn_tc_kernel<128>(const AttnArgs, const __grid_constant__ CUtensorMap,
                                                  const __grid_constant__ CUtensorMap,
                                                  const __grid_constant__ CUtensorMap);

// Host launcher (declared in attn_common.cuh).
template <int D>
int launch_attn_tc(const AttnArgs &args, int max_prefix, int T, const CUtensorMap &tmq,
                   const CUtensorMap &tmk, const CUtensorMap &tmv, int num_sms, cudaStream_t stream) {
  using C = TcCfg<D>;
  auto kernel = tree_attn_tc_kernel<D>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
        cudaSuccess)
      return SPEC_ERR_CUDA;
    configured = true;
  }
  const int max_nodes = T < SPEC_MAX_TREE_NODES ? T : SPEC_MAX_TREE_NODES;
  const int rowblocks = (max_nodes * args.G + kTcRows - 1) / kTcRows;
  const long long max_keys = static_cast<long long>(max_prefix) + max_nodes;
  const long long tiles_max = (max_keys + kKeyTile - 1) / kKeyTile;
  const long long units = static_cast<long long>(rowblocks) * args.B * args.Hkv;
  if (units > 65535) return SPEC_ERR_SHAPE;
  // Pick the split count that minimises (waves x tiles per CTA), one CTA/SM.
  int cs = 1;
  long long best = -1;
  for (int c = 1; c <= 8; c *= 2) {
    if (c > 1 && tiles_max < 2 * c) break;
    const long long waves = (units * c + num_sms - 1) / num_sms;
    const long long cost = waves * ((tiles_max + c - 1) / c) + (c > 1 ? 1 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      cs = c;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, rowblocks, static_cast<unsigned>(args.B * args.Hkv));
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args, tmq, tmk, tmv) == cudaSuccess ? SPEC_OK
                                                                             : SPEC_ERR_CUDA;
}

template int launch_attn_tc<64>(const AttnArgs &, int, int, const CUtensorMap &, const CUtensorMap &,
                                const CUtensorMap &, int, cudaStream_t);
template int launch_attn_tc<128>(const AttnArgs &, int, int, const CUtensorMap &, const CUtensorMap &,
                                 const CUtensorMap &, int, cudaStream_t);

}  // namespace spec
