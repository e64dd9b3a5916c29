// Steps A2 and A3 on the 5th-generation tensor cores (tcgen05), bf16 in,
// fp32 accumulate.
//
// SpecInfer developer article §2.1, tree_attention snippet (masked scores,
// softmax, times V); SpecInfer news write-up "Token 樹驗證器" (tree K/V
// appended to the cache depth-first, mask restricted to the node's ancestors).
//
// One CTA = one key split x one block of query rows x one (request, KV head).
// Rows are (node, head-in-group) pairs, so one K/V tile feeds all G query
// heads of the KV head.  Warp roles:
//   warp 0      TMA producer: the Q block once, then 64-key K and V tiles
//               (128-byte swizzle) into a ring of stages.
//   warp 1      allocates TMEM; one thread issues S_i = Q K_i^T
//               (M=128, N=64, K=D, into TMEM S[i%3]) as soon as K_i has
//               landed and S[i%3] is free, so the softmax of one tile
//               overlaps the QK^T of the next ones.
//   warp 2      one thread issues O += P_i V_i (M=128, N=D, K=64, TMEM O)
//               as soon as P_i is written: two issuing threads, so neither
//               kind of MMA waits behind the other's issue.
//   warps 3+    four threads per TMEM lane (= query row), one per quarter of
//               the tile's keys (16 softmax warps for 128-row blocks, 8 for
//               packed blocks): read S from TMEM, mask with the node's
//               ancestor bits, share the row max, online softmax with a
//               lazily moved reference max (the stored O is rescaled only
//               when a row's max grows by more than 2^8), write P as bf16
//               high and remainder parts (P V then keeps about 16
//               significant bits of every weight): into TMEM for 128-row
//               blocks, whose P V takes its A operand from TMEM, into shared
//               memory for packed blocks.
// Blocks of at most 64 rows (PACKED) load their Q rows twice (rows 0-63 and
// 64-127 of the MMA), so TMEM lanes r and r + 64 both hold S row r: four
// threads per row spread the softmax over all four SM sub-partitions, and
// the remainder part of P goes to P rows 64-127, so one 4-MMA P V pass per
// tile leaves the high part in lanes 0-63 and the remainder in 64-127 (added
// at the end).  The single P operand leaves room for a 4-stage K/V ring.
// Outputs leave through a shared-memory staging buffer so global stores are
// coalesced.  The key splits of a block form one thread-block cluster: each
// split stages its (O, m, l) rows in shared memory, and after a cluster
// barrier sends each row's owner that owner's rows with one bulk
// shared-to-shared copy; owners merge locally (a cluster stays on one die,
// so no cross-die L2 round trip is involved).
#include <cuda.h>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "tcgen05.cuh"

namespace spec {

constexpr int kTcRows = 128;
constexpr float kRescaleLog2 = 8.f;

template <int D, bool PACKED>
struct TcCfg {
  // packed blocks keep P in shared memory (their remainder rows come from other
  // threads' lanes); 128-row blocks write P into TMEM, which frees room for a
  // deeper K/V ring
  static constexpr int kStages = PACKED ? 4 : 5;
  static constexpr int kBoxes = D / 64;
  static constexpr int kLoadRows = PACKED ? kTcRows / 2 : kTcRows;  // rows one Q load brings
  static constexpr int kQLoadBytes = kLoadRows * 128;
  static constexpr int kQChunkBytes = kTcRows * 128;   // smem per 64-dim chunk of the Q block
  static constexpr int kQBytes = kTcRows * D * 2;
  static constexpr int kKVBoxBytes = kKeyTile * 128;
  static constexpr int kTileBytes = kKeyTile * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kPBytes = kTcRows * kKeyTile * 2;   // one 128-row bf16 P operand
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffP = kOffKV + kStages * kStageBytes;
  static constexpr int kPSmem = PACKED ? 2 * kPBytes : 0;   // P in shared memory (packed)
  static constexpr int kSmem = kOffP + kPSmem + 1024;
  // softmax warps: four threads (key quarters) per S row; packed blocks hold
  // 64 rows twice, so 8 warps cover them, 128-row blocks take 16
  static constexpr int kSoftmaxWarps = PACKED ? 8 : 16;
  static constexpr int kThreads = 32 * (3 + kSoftmaxWarps);   // TMA, S issuer, P V issuer, softmax
  static constexpr int kParts = 4;                          // threads per row (key parts)
  static constexpr int kKeysPer = kKeyTile / kParts;        // keys per thread per tile
  static constexpr int kOCols = PACKED ? D / 2 : D / 4;     // O columns one thread reads out
  static constexpr int kStage = D + 4;                      // floats per staged output row
  static constexpr int kSBufs = 3;                          // S tiles in flight in TMEM
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;                      // S buffers: 3 x 64 columns
  static constexpr uint32_t kColO = 256;                    // O: D columns
  static constexpr uint32_t kColP = 384;                    // 128-row P: 2 x (32 high + 32 remainder)
  static_assert(!PACKED || kTcRows / 2 * D * 4 <= kPSmem,
                "packed remainder exchange fits the P buffers");
  static_assert(PACKED || kColO + D <= kColP, "O and P columns are disjoint");
  static_assert(kTcRows * kStage * 4 <= kStages * kStageBytes, "output staging fits the K/V ring");
  // staged rows plus the receive slots of the split merge, in the ring and P buffers
  static_assert((2 * (PACKED ? kTcRows / 2 : kTcRows) + 8) * kStage * 4 <=
                    kStages * kStageBytes + kPSmem,
                "split-merge buffers fit");
  static_assert(kOffP == kOffKV + kStages * kStageBytes, "ring and P buffers are contiguous");
  static_assert(kSmem <= 227 * 1024 - 8192, "shared memory budget");
};

constexpr int kTcMaxSplits = 8;
constexpr int kEarlyTiles = 2;   // K/V tiles requested with Q, before tile 0 lands
// K/V tiles of a split prefetched into L2 before the PDL wait: one, so that
// every split's first tile arrives ahead of the rest of the ring's initial
// fill (a deeper prefetch queues all of them together in HBM).
constexpr int kPrefetchTiles = 1;



// L2 prefetch of one tile of a tensor map (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_4d(const void *tmap, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const void *tmap, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// N consecutive TMEM columns of this thread's lane into registers (N a
// multiple of 16), and the same columns scaled in place.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&out)[N]) {
  static_assert(N % 16 == 0, "16-column granularity");
  if constexpr (N % 32 == 0) {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
      float o[32];
      tc::ld32(taddr + c * 32, o);
      tc::wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) out[c * 32 + e] = o[e];
    }
  } else {
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
      float o[16];
      tc::ld16(taddr + c * 16, o);
      tc::wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) out[c * 16 + e] = o[e];
    }
  }
}

template <int N>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, float alpha) {
  static_assert(N % 16 == 0, "16-column granularity");
  if constexpr (N % 32 == 0) {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
      float o[32];
      tc::ld32(taddr + c * 32, o);
      tc::wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] *= alpha;
      tc::st32(taddr + c * 32, o);
    }
  } else {
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
      float o[16];
      tc::ld16(taddr + c * 16, o);
      tc::wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] *= alpha;
      tc::st16(taddr + c * 16, o);
    }
  }
  tc::wait_st();
}

__device__ __forceinline__ int ld_volatile_shared(const int *p) {
  int v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_volatile_shared(int *p, int v) {
  asm volatile("st.volatile.shared.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<const uint32_t *>(&v);
}

template <int D, bool PACKED>
__global__ void __launch_bounds__(TcCfg<D, PACKED>::kThreads, 1)
tree_attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  using C = TcCfg<D, PACKED>;
  constexpr int NS = C::kStages;
  constexpr int KP = C::kKeysPer;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[NS], bar_empty[NS];
  __shared__ __align__(8) uint64_t bar_q, bar_s[3], bar_p[2], bar_o[2];
  __shared__ uint32_t s_tmem;
  __shared__ float x_max[2][C::kParts][kTcRows];   // [tile parity][key part][row]
  __shared__ float x_l[C::kParts][kTcRows];
  __shared__ __align__(8) uint64_t bar_m;          // key splits: the peers' rows have arrived
  __shared__ int s_timeout;
  __shared__ int s_pv_issued;                        // P V products issued so far (warp 2)
  __shared__ int s_par[SPEC_MAX_TREE_NODES];         // the request's parents (no mask array)

  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const int CS = static_cast<int>(gridDim.x);   // the key splits of a block form one cluster
  const int split = static_cast<int>(blockIdx.x);
  const int rb = blockIdx.y;
  const int b = blockIdx.z / a.Hkv;
  const int g = blockIdx.z % a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- set-up that reads no global memory, overlapping the previous kernel
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_q, 1);
    mbar_init(&bar_m, 1);
    for (int j = 0; j < 3; ++j) mbar_init(&bar_s[j], 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&bar_p[j], C::kSoftmaxWarps);
      mbar_init(&bar_o[j], 1);
    }
    fence_barrier_init();
    s_timeout = 0;
    s_pv_issued = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    if (a.prefetch_keys > 0) {
      // One request whose key count the host knows: this split's first
      // tile, and its Q rows, are prefetched into L2 while the previous
      // kernel still runs.  A prefetch only warms L2, which every write of
      // the previous kernel updates, so it can never serve stale data; if the
      // request's real key count differs, the prefetched lines are unused.
      const int tiles = (a.prefetch_keys + kKeyTile - 1) / kKeyTile;
      const int per = (tiles + CS - 1) / CS;
      const int t0 = split * per;
      const int nt = min(kPrefetchTiles, min(t0 + per, tiles) - t0);
      for (int i = 0; i < nt; ++i)
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_prefetch_l2_4d(&tmk, bx * 64, (t0 + i) * kKeyTile, g, 0);
          tma_prefetch_l2_4d(&tmv, bx * 64, (t0 + i) * kKeyTile, g, 0);
        }
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) tma_prefetch_l2_3d(&tmq, bx * 64, g * a.G, rb * kTcRows / a.G);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(&s_tmem, C::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  pdl_wait();

  const ReqGeom R = request_geometry(a, b);
  const int rows_total = R.n * a.G;
  const int row0 = rb * kTcRows;
  const int rows_here = min(kTcRows, rows_total - row0);
  // Whole-block exits are uniform across the cluster (same request and row
  // block); the block frees its tensor memory first.
  const bool bad_block = PACKED && !R.err && row0 < rows_total && rows_here > kTcRows / 2;
  if (R.err || row0 >= rows_total || bad_block) {
    if (R.err && tid == 0 && split == 0 && rb == 0 && g == 0) report(a.status, b, R.err);
    if (bad_block && tid == 0) report(a.status, b, SPEC_ERR_SHAPE);  // launch contract broken
    if (warp == 1) {
      __syncwarp();
      tc::tmem_dealloc(tmem, C::kTmemCols);
    }
    return;
  }
  const int tiles_total = (R.keys + kKeyTile - 1) / kKeyTile;
  const int per = (tiles_total + CS - 1) / CS;
  const int t0 = split * per;
  const int ntiles = max(0, min(t0 + per, tiles_total) - t0);

  // softmax-thread geometry (warps 3 and up).  TMEM lane r = 32 * quad +
  // lane.  128-row blocks: row r, four threads (key quarters) per row, each
  // reading out a quarter of the row's O.  Packed blocks: the Q block is
  // loaded twice, so lanes r and r + 64 hold the same S row; four threads
  // (key quarters) per row, lanes 64-127 accumulate the remainder part of
  // P V, and each thread reads out half of its lane's O.
  const int quad = warp & 3;
  const int half = (warp - 3) >> 2;                  // packed: 0..1; otherwise 0..3
  const int part = PACKED ? ((quad >> 1) * 2 + half) : half;
  const int srow = PACKED ? ((quad & 1) * 32 + lane) : (quad * 32 + lane);
  const bool row_ok = srow < rows_here;
  const bool lanes_live = warp >= 3 && (PACKED ? (quad & 1) : quad) * 32 < rows_here;
  const bool lo_lane = PACKED && quad >= 2;          // holds the remainder part of P V
  const bool owner = warp >= 3 && !lo_lane;          // assembles the row's final O
  const int ocol = PACKED ? half * (D / 2) : part * (D / 4);   // this thread's O columns
  const bool tail_writer = PACKED ? half == 0 : part == 0;
  constexpr int kOC = C::kOCols;
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  float o_keep[kOC];
  float m_used = -INFINITY, l_part = 0.f, l_row = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      mbar_arrive_expect_tx(&bar_q, C::kQBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_3d(smem + C::kOffQ + bx * C::kQChunkBytes, &tmq, &bar_q, bx * 64, g * a.G,
                    R.lo + row0 / a.G);
        if (PACKED)  // the same 64 rows again into rows 64-127
          tma_load_3d(smem + C::kOffQ + bx * C::kQChunkBytes + C::kQLoadBytes, &tmq, &bar_q,
                      bx * 64, g * a.G, R.lo + row0 / a.G);
      }
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        // Q and the first two tiles go first: every CTA's first tile then
        // lands ahead of the rest of the ring's initial fill, so the first S
        // starts earlier; the other stages are requested once tile 0 is in.
        if (i == kEarlyTiles && !mbar_wait(&bar_full[0], 0)) {
          s_timeout = 1;
          break;
        }
        if (i >= NS && !mbar_wait(&bar_empty[st], ((i / NS) - 1) & 1)) {
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
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1 issues S_i = Q K_i^T, warp 2 issues O += P_j V_j: two
    // instruction streams, so neither kind waits behind the other's issue.
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcRows, kKeyTile, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kTcRows, D, 0, 1);
      bool ok = true;
      // Descriptors: one base per operand kind, the start address (bits
      // [0, 14), in 16-byte units) advanced by adding the offset; every
      // shared-memory address stays below 256 KB, so the field never carries.
      const uint64_t qd0 = tc::smem_desc_sw128(sb + C::kOffQ, 16, 1024);
      const uint64_t kd0 = tc::smem_desc_sw128(sb + C::kOffKV, 16, 1024);
      const uint64_t vd0 = tc::smem_desc_sw128(sb + C::kOffKV + C::kTileBytes, C::kKVBoxBytes, 1024);
      auto issue_s = [&](int i) {
        const int st = i % NS;
        tc::fence_after_sync();
        const uint64_t kd = kd0 + static_cast<uint64_t>((st * C::kStageBytes) >> 4);
        const uint32_t sc = tmem + C::kColS + (i % C::kSBufs) * kKeyTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * C::kQChunkBytes + (ks & 3) * 32) >> 4;
          const uint32_t koff = ((ks >> 2) * C::kKVBoxBytes + (ks & 3) * 32) >> 4;
          tc::mma_bf16(sc, qd0 + off, kd + koff, idS, ks > 0);
        }
        tc::commit(&bar_s[i % C::kSBufs]);
      };
      auto issue_pv = [&](int j) {
        const int st = j % NS;
        tc::fence_after_sync();
        const uint64_t vd = vd0 + static_cast<uint64_t>((st * C::kStageBytes) >> 4);
        if constexpr (PACKED) {
          const uint64_t pd =
              tc::smem_desc_sw128(sb + C::kOffP, 16, 1024) + static_cast<uint64_t>(((j & 1) * C::kPBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk)
            tc::mma_bf16(tmem + C::kColO, pd + (kk * 32 >> 4), vd + (kk * 16 * 128 >> 4), idO, (j | kk) != 0);
        } else {
          // A = P from TMEM: high part in columns [0, 32) of the buffer, the
          // remainder in [32, 64); eight columns per 16 keys
          const uint32_t pt = tmem + C::kColP + (j & 1) * kKeyTile;
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
            for (int kk = 0; kk < kKeyTile / 16; ++kk)
              tc::mma_bf16_ts(tmem + C::kColO, pt + pp * 32 + kk * 8, vd + (kk * 16 * 128 >> 4), idO,
                              (j | pp | kk) != 0);
          }
        }
        tc::commit(&bar_o[j & 1]);
        tc::commit(&bar_empty[st]);
      };
      if (warp == 1) {
        // S_i goes into TMEM buffer i % 3 once tile i's K/V has landed and the
        // softmax has read S_{i-3}: P V of tile i - 3 has been issued (its P
        // arrived), which warp 2 publishes in s_pv_issued.
        ok = ok && mbar_wait(&bar_q, 0);
        for (int i = 0; ok && i < ntiles; ++i) {
          if (i >= C::kSBufs) {
            const uint64_t t0 = global_ns();
            for (uint32_t it = 1; ld_volatile_shared(&s_pv_issued) < i - C::kSBufs + 1; ++it)
              if ((it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
                ok = false;
                break;
              }
          }
          if (ok && !mbar_wait(&bar_full[i % NS], (i / NS) & 1)) ok = false;
          if (ok) issue_s(i);
        }
      } else {
        // P_j V_j goes once P_j has arrived (its K/V landed before S_j)
        for (int j = 0; ok && j < ntiles; ++j) {
          if (!mbar_wait(&bar_p[j & 1], (j >> 1) & 1)) {
            ok = false;
            break;
          }
          issue_pv(j);
          st_volatile_shared(&s_pv_issued, j + 1);
        }
      }
      if (!ok) s_timeout = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    uint4 msk = make_uint4(0, 0, 0, 0);
    if (a.mask) {
      if (lanes_live && row_ok && in_bounds(R.lo + (row0 + srow) / a.G, a.T, a.status, b))
        msk = clip_mask(__ldg(a.mask + R.lo + (row0 + srow) / a.G), R.n);
    } else {
      // no mask array: the softmax warps stage the request's parents, and
      // each thread walks its row's node to the root (the first S tile is
      // still on its way)
      for (int i = tid - 96; i < R.n; i += 32 * C::kSoftmaxWarps)
        s_par[i] = in_bounds(R.lo + i, a.T, a.status, b) ? __ldg(a.parents + R.lo + i) : -2;
      named_bar_sync(2, 32 * C::kSoftmaxWarps);
      bool bad = false;
      if (lanes_live && row_ok)
        msk = ancestor_mask([&](int i) { return s_par[i]; }, (row0 + srow) / a.G, &bad);
      if (bad) report(a.status, b, SPEC_ERR_BAD_PARENT);
    }
    const float sl2 = a.scale_log2;
    bool ok = true;
    // A timed-out wait clears `ok` and later waits are skipped, but the loop
    // runs to the end so every softmax warp meets every named barrier.
    for (int i = 0; i < ntiles; ++i) {
      if (ok && !mbar_wait(&bar_s[i % C::kSBufs], (i / C::kSBufs) & 1)) ok = false;
      __syncwarp();
      tc::fence_after_sync();
      const int key0 = (t0 + i) * kKeyTile;
      const int st = i % NS;
      if (key0 + kKeyTile > R.keys) {
        // V rows past the request's last key may hold anything: zero them so
        // their zero weights contribute exact zeros.
        const int valid = R.keys - key0;
        const int chunks = (kKeyTile - valid) * C::kBoxes * 8;
        uint8_t *vrow = smem + C::kOffKV + st * C::kStageBytes + C::kTileBytes;
        for (int c = tid - 96; c < chunks; c += 32 * C::kSoftmaxWarps) {
          const int row = valid + c / (C::kBoxes * 8);
          const int rest = c % (C::kBoxes * 8);
          *reinterpret_cast<uint4 *>(vrow + (rest >> 3) * C::kKVBoxBytes + row * 128 +
                                     (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      float s[KP];
      bool want = false;
      if (lanes_live) {
        const uint32_t scol = trow + C::kColS + (i % C::kSBufs) * kKeyTile + KP * part;
        if constexpr (KP == 32) {
          tc::ld32(scol, *reinterpret_cast<float(*)[32]>(s));
        } else {
          tc::ld16(scol, *reinterpret_cast<float(*)[16]>(s));
        }
        tc::wait_ld();
        const int kbase = key0 + KP * part;
        if (kbase + KP > R.L) {
#pragma unroll
          for (int j = 0; j < KP; ++j)
            if (!key_visible(kbase + j, R.L, R.keys, msk)) s[j] = -INFINITY;
        }
        float mt = s[0];
#pragma unroll
        for (int j = 1; j < KP; ++j) mt = fmaxf(mt, s[j]);
        x_max[i & 1][part][srow] = mt;
        want = row_ok && (mt * sl2 > m_used + kRescaleLog2);
      }
      // one barrier: every part's maximum is visible, and whether any row of
      // the block moves its reference max
      const bool any_resc = named_bar_or(2, 32 * C::kSoftmaxWarps, want);
      if (any_resc) {
        float mt = -INFINITY;
        if (lanes_live && row_ok) {
#pragma unroll
          for (int q = 0; q < C::kParts; ++q) mt = fmaxf(mt, x_max[i & 1][q][srow]);
          mt *= sl2;
        }
        const bool resc = row_ok && lanes_live && (mt > m_used + kRescaleLog2);
        const float m_new = resc ? mt : m_used;
        const float alpha = !resc ? 1.f : (m_used == -INFINITY ? 0.f : exp2f(m_used - m_new));
        if (i > 0 && lanes_live) {
          // O holds the products of tiles < i: wait for the last of them,
          // then rescale this thread's columns of its TMEM lane in place.
          if (ok && !mbar_wait(&bar_o[(i - 1) & 1], ((i - 1) >> 1) & 1)) ok = false;
          __syncwarp();
          tc::fence_after_sync();
          tmem_scale_cols<kOC>(trow + C::kColO + ocol, alpha);
        }
        l_part *= alpha;
        m_used = m_new;
      }
      if (lanes_live) {
        const float nbase = (m_used == -INFINITY) ? 0.f : -m_used;
        // the tile's weights first, in place, so they are ready while the P
        // buffer may still be busy
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < KP; ++j) {
          s[j] = fast_exp2(fmaf(s[j], sl2, nbase));
          psum += s[j];
        }
        // the P buffer of this parity is free once the P V of tile i-2 is done
        if (ok && i >= 2 && !mbar_wait(&bar_o[i & 1], ((i - 2) >> 1) & 1)) ok = false;
        __syncwarp();
        if constexpr (PACKED) {
          uint8_t *pbuf = smem + C::kOffP + (i & 1) * C::kPBytes;
          uint8_t *prow_hi = pbuf + srow * 128;
          uint8_t *prow_lo = pbuf + (srow + kTcRows / 2) * 128;
#pragma unroll
          for (int cc = 0; cc < KP / 8; ++cc) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p0 = s[cc * 8 + 2 * e], p1 = s[cc * 8 + 2 * e + 1];
              const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
              const float2 hf = __bfloat1622float2(h);
              hi[e] = bf16x2_bits(h);
              lo[e] = bf16x2_bits(__floats2bfloat162_rn(p0 - hf.x, p1 - hf.y));
            }
            const int off = (((KP / 8) * part + cc) ^ (srow & 7)) << 4;   // (srow + 64) & 7 == srow & 7
            *reinterpret_cast<uint4 *>(prow_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(prow_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        } else {
          // P into this thread's TMEM lane: its 16 keys are columns
          // [8 part, 8 part + 8) of the high and of the remainder half
          static_assert(PACKED || KP == 16, "128-row blocks: 16 keys per thread");
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float p0 = s[2 * e], p1 = s[2 * e + 1];
            const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
            const float2 hf = __bfloat1622float2(h);
            hi[e] = bf16x2_bits(h);
            lo[e] = bf16x2_bits(__floats2bfloat162_rn(p0 - hf.x, p1 - hf.y));
          }
          const uint32_t pt = trow + C::kColP + (i & 1) * kKeyTile + 8 * part;
          tc::st8(pt, hi);
          tc::st8(pt + 32, lo);
          tc::wait_st();
        }
        l_part += psum;
      }
      // P (packed blocks) and the zeroed V rows of a tail tile are generic
      // shared-memory stores that the P V product reads through the async
      // proxy: order them before the arrival that releases the issuer.
      if (PACKED || key0 + kKeyTile > R.keys) fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[i & 1]);
    }
    if (!ok) s_timeout = 1;
    // ---- epilogue: O rows out of TMEM.  Every softmax warp waits for the
    //      last P V before any thread reuses the K/V ring or the P buffers; a
    //      thread whose waits ran out writes no shared memory (copies may
    //      still land there).
    if (ntiles > 0) {
      if (ok && !mbar_wait(&bar_o[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) {
        ok = false;
        s_timeout = 1;
      }
      __syncwarp();
      tc::fence_after_sync();
    }
#pragma unroll
    for (int e = 0; e < kOC; ++e) o_keep[e] = 0.f;
    if (ok && lanes_live && ntiles > 0) tmem_load_cols<kOC>(trow + C::kColO + ocol, o_keep);
    // [64 rows][D] floats in the free P buffers; 16-byte chunks swizzled by
    // row so that eight consecutive rows hit eight different bank groups
    float *xo = reinterpret_cast<float *>(smem + C::kOffP);
    auto xo_at = [&](int e) -> float4 * {
      const int chunk = (ocol + e) >> 2;
      return reinterpret_cast<float4 *>(xo + srow * D) + (chunk ^ (srow & 7));
    };
    if (ok && PACKED && lo_lane && row_ok) {
#pragma unroll
      for (int e = 0; e < kOC; e += 4)
        *xo_at(e) = make_float4(o_keep[e], o_keep[e + 1], o_keep[e + 2], o_keep[e + 3]);
    }
    if (warp >= 3) x_l[part][srow] = l_part;
    named_bar_sync(2, 32 * C::kSoftmaxWarps);
    if (ok && owner && row_ok) {
#pragma unroll
      for (int q = 0; q < C::kParts; ++q) l_row += x_l[q][srow];
      if (PACKED) {
#pragma unroll
        for (int e = 0; e < kOC; e += 4) {
          const float4 v = *xo_at(e);
          o_keep[e] += v.x;
          o_keep[e + 1] += v.y;
          o_keep[e + 2] += v.z;
          o_keep[e + 3] += v.w;
        }
      }
      // stage the row, O then (m, l), for coalesced stores or the split
      // merge (the K/V ring is free)
      float *stg = reinterpret_cast<float *>(smem + C::kOffKV) + srow * C::kStage;
#pragma unroll
      for (int e = 0; e < kOC; e += 4)
        *reinterpret_cast<float4 *>(stg + ocol + e) =
            make_float4(o_keep[e], o_keep[e + 1], o_keep[e + 2], o_keep[e + 3]);
      if (tail_writer) *reinterpret_cast<float2 *>(stg + D) = make_float2(ntiles > 0 ? m_used : -INFINITY, l_row);
      fence_proxy_async_smem();  // the rows may leave by bulk copy
    }
  }

  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
  // A wait that ran out anywhere in the CTA: report it and write no output
  // row of the block (with key splits, no CTA of the cluster writes one).
  const bool timed_out = s_timeout != 0;
  if (timed_out && tid == 0) report(a.status, b, SPEC_ERR_TIMEOUT);
  const float *stg = reinterpret_cast<const float *>(smem + C::kOffKV);
  if (CS == 1) {
    if (timed_out) return;
    // ---- final rows, 8 bf16 per thread, consecutive threads on one row
    const int nv = rows_here * (D / 8);
    for (int idx = tid; idx < nv; idx += C::kThreads) {
      const int lr = idx / (D / 8), c8 = idx % (D / 8);
      const float inv = 1.f / stg[lr * C::kStage + D + 1];
      const float4 v0 = *reinterpret_cast<const float4 *>(stg + lr * C::kStage + c8 * 8);
      const float4 v1 = *reinterpret_cast<const float4 *>(stg + lr * C::kStage + c8 * 8 + 4);
      uint4 pk;
      pk.x = bf16x2_bits(__floats2bfloat162_rn(v0.x * inv, v0.y * inv));
      pk.y = bf16x2_bits(__floats2bfloat162_rn(v0.z * inv, v0.w * inv));
      pk.z = bf16x2_bits(__floats2bfloat162_rn(v1.x * inv, v1.y * inv));
      pk.w = bf16x2_bits(__floats2bfloat162_rn(v1.z * inv, v1.w * inv));
      const int rr = row0 + lr;
      if (!in_bounds(R.lo + rr / a.G, a.T, a.status, b)) continue;
      *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.o) +
                                 (static_cast<size_t>(R.lo + rr / a.G) * a.Hq + g * a.G + rr % a.G) * D +
                                 c8 * 8) = pk;
    }
    return;
  }
  // ---- key splits.  CTA `split` owns rows [split * rpr, ...) of the block.
  //      After a cluster barrier (every split has staged its rows, every K/V
  //      ring is free), each CTA sends every owner that owner's rows with one
  //      bulk shared-to-shared copy into the owner's receive slot [sender],
  //      completing on the owner's barrier; each owner merges locally.
  const int rpr = (rows_here + CS - 1) / CS;
  auto own_range = [&](int r, int &r0, int &rn) {
    r0 = min(rows_here, r * rpr);
    rn = min(rows_here, r0 + rpr) - r0;
  };
  int own0, own_n;
  own_range(split, own0, own_n);
  float *recv = const_cast<float *>(stg) + rows_here * C::kStage;   // [CS][rpr][kStage]
  cluster_sync_all();
  // Every CTA sends its rows even after a timeout (the byte counts complete
  // the owners' barriers; the rows are then unused), and reads whether any
  // CTA of the cluster timed out: every s_timeout is final after the barrier.
  __shared__ int s_cluster_timeout;
  if (tid == 0) {
    if (own_n > 0) mbar_arrive_expect_tx(&bar_m, static_cast<uint32_t>((CS - 1) * own_n * C::kStage * 4));
    for (int r = 0; r < CS; ++r) {
      int r0, rn;
      own_range(r, r0, rn);
      if (r == split || rn <= 0) continue;
      bulk_copy_s2s(peer_addr(recv + split * rpr * C::kStage, r), smem_addr(stg + r0 * C::kStage),
                    static_cast<uint32_t>(rn * C::kStage * 4), peer_addr(&bar_m, r));
    }
    int any = timed_out ? 1 : 0;
    for (int r = 0; r < CS; ++r)
      if (r != split) any |= ld_peer_s32(peer_addr(&s_timeout, static_cast<uint32_t>(r)));
    s_cluster_timeout = any;
  }
  if (own_n > 0 && !mbar_wait(&bar_m, 0) && tid == 0) {
    report(a.status, b, SPEC_ERR_TIMEOUT);
    s_cluster_timeout = 1;
  }
  __syncthreads();
  cluster_arrive_relaxed();  // everything addressed to this CTA has arrived
  if (s_cluster_timeout) {
    cluster_wait();   // no CTA leaves while a copy may still read its rows
    return;
  }
  {
    constexpr int kE = D / 8;   // columns per task
    const int ntask = own_n * 8;
    for (int task = tid; task < ntask; task += C::kThreads) {
      const int j = task >> 3;
      const int lr = own0 + j;
      const int col0 = (task & 7) * kE;
      auto part = [&](int q) -> const float * {
        return q == split ? stg + lr * C::kStage : recv + (q * rpr + j) * C::kStage;
      };
      float M = -INFINITY;
      for (int q = 0; q < CS; ++q) M = fmaxf(M, part(q)[D]);
      float acc[kE];
#pragma unroll
      for (int e = 0; e < kE; ++e) acc[e] = 0.f;
      float L = 0.f;
      for (int q = 0; q < CS; ++q) {
        const float *row = part(q);
        const float2 ml = *reinterpret_cast<const float2 *>(row + D);
        if (ml.x == -INFINITY) continue;
        const float w = exp2f(ml.x - M);
        L += w * ml.y;
#pragma unroll
        for (int q4 = 0; q4 < kE / 4; ++q4) {
          const float4 v = *reinterpret_cast<const float4 *>(row + col0 + 4 * q4);
          acc[4 * q4 + 0] += w * v.x;
          acc[4 * q4 + 1] += w * v.y;
          acc[4 * q4 + 2] += w * v.z;
          acc[4 * q4 + 3] += w * v.w;
        }
      }
      const float inv = 1.f / L;
      const int rr = row0 + lr;
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.o) +
                           (static_cast<size_t>(R.lo + rr / a.G) * a.Hq + g * a.G + rr % a.G) * D + col0;
      const bool store = in_bounds(R.lo + rr / a.G, a.T, a.status, b);
#pragma unroll
      for (int q8 = 0; q8 < kE / 8 && store; ++q8) {
        uint4 pk;
        pk.x = bf16x2_bits(__floats2bfloat162_rn(acc[q8 * 8 + 0] * inv, acc[q8 * 8 + 1] * inv));
        pk.y = bf16x2_bits(__floats2bfloat162_rn(acc[q8 * 8 + 2] * inv, acc[q8 * 8 + 3] * inv));
        pk.z = bf16x2_bits(__floats2bfloat162_rn(acc[q8 * 8 + 4] * inv, acc[q8 * 8 + 5] * inv));
        pk.w = bf16x2_bits(__floats2bfloat162_rn(acc[q8 * 8 + 6] * inv, acc[q8 * 8 + 7] * inv));
        *reinterpret_cast<uint4 *>(dst + q8 * 8) = pk;
      }
    }
  }
  cluster_wait();  // no CTA leaves while a copy may still read its rows
}

// Split plan: the split count (cluster size) that minimises the time of the
// launch at one CTA per SM, in units of one key tile: waves x (tiles per CTA
// + a CTA's fixed ramp-up and epilogue, about 4 tiles, + the split merge,
// about 3 tiles).
void plan_attn_tc(int B, int T, int Hkv, int G, int max_prefix, int num_sms, int *cs_out,
                  int *rowblocks_out) {
  const int max_nodes = T < SPEC_MAX_TREE_NODES ? T : SPEC_MAX_TREE_NODES;
  const int rowblocks = (max_nodes * G + kTcRows - 1) / kTcRows;
  const long long max_keys = static_cast<long long>(max_prefix) + max_nodes;
  const long long tiles_max = (max_keys + kKeyTile - 1) / kKeyTile;
  const long long units = static_cast<long long>(rowblocks) * B * Hkv;
  int cs = 1;
  long long best = -1;
  for (int c = 1; c <= kTcMaxSplits; ++c) {
    if (c > 1 && tiles_max < 2 * c) break;
    const long long waves = (units * c + num_sms - 1) / num_sms;
    const long long cost = waves * ((tiles_max + c - 1) / c + 4 + (c > 1 ? 3 : 0));
    if (best < 0 || cost < best) {
      best = cost;
      cs = c;
    }
  }
  *cs_out = cs;
  *rowblocks_out = rowblocks;
}

template <int D, bool PACKED>
static int launch_tc(const AttnArgs &args, const CUtensorMap &tmq, const CUtensorMap &tmk,
                     const CUtensorMap &tmv, int cs, int rowblocks, cudaStream_t stream) {
  using C = TcCfg<D, PACKED>;
  auto kernel = tree_attn_tc_kernel<D, PACKED>;
  static std::atomic<size_t> granted[kMaxDevices];
  if (!allow_dynamic_smem(kernel, C::kSmem, granted)) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, rowblocks, static_cast<unsigned>(args.B * args.Hkv));
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attribute(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args, tmq, tmk, tmv) == cudaSuccess ? SPEC_OK
                                                                             : SPEC_ERR_CUDA;
}

int launch_attn_tc(const AttnArgs &args, int max_prefix, int T, const CUtensorMap &tmq,
                   const CUtensorMap &tmk, const CUtensorMap &tmv, bool packed, int num_sms,
                   cudaStream_t stream) {
  int cs, rowblocks;
  plan_attn_tc(args.B, T, args.Hkv, args.G, max_prefix, num_sms, &cs, &rowblocks);
  if (static_cast<long long>(rowblocks) * args.B * args.Hkv > 65535) return SPEC_ERR_SHAPE;
  if (args.D == 128)
    return packed ? launch_tc<128, true>(args, tmq, tmk, tmv, cs, rowblocks, stream)
                  : launch_tc<128, false>(args, tmq, tmk, tmv, cs, rowblocks, stream);
  return packed ? launch_tc<64, true>(args, tmq, tmk, tmv, cs, rowblocks, stream)
                : launch_tc<64, false>(args, tmq, tmk, tmv, cs, rowblocks, stream);
}

}  // namespace spec
