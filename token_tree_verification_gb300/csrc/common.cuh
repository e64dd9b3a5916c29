// Device helpers shared by the library's kernels: status reporting, bounded
// mbarrier waits, TMA tile loads, cluster/DSMEM access and the counter-based
// generator.  sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/spec_tree.h"

namespace spec {

// A bounded wait gives up and reports SPEC_ERR_TIMEOUT after this many
// nanoseconds (2 s), far beyond any legitimate wait in these kernels.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  Kernels launched with the
// programmatic-serialization attribute may start before the previous kernel
// in the stream has finished: they signal their own dependents at once, do
// only set-up (barriers, tensor-memory allocation) before pdl_wait(), and
// touch no global memory before it; pdl_wait() returns once the previous
// grid has completed and its writes are visible (at once without a
// programmatic predecessor).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

inline void pdl_attribute(cudaLaunchAttribute &attr) {
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
}

// ---------------------------------------------------------------- host state
// What a launcher caches about the GPU (a kernel's shared-memory limit, the
// SM count) belongs to one device, so it is kept per device ordinal.
constexpr int kMaxDevices = 256;

inline int current_device() {
  int dev = 0;
  return (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

// SMs of the current device (launch plans size grids by it); 152 (GB300)
// when no device can be queried.
inline int sm_count() {
  static std::atomic<int> n[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 152;
  int v = n[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return 152;
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// A kernel needs its dynamic shared-memory limit raised before a launch with
// more than 48 KB, on each device it runs on.  `granted[dev]` holds the
// largest limit set on device dev; the limit only ever grows, and changes
// are serialised, so a concurrent launch never sees it lowered.
template <typename Kernel>
inline bool allow_dynamic_smem(Kernel kernel, size_t bytes, std::atomic<size_t> *granted) {
  const int dev = current_device();
  if (dev < 0) return false;
  if (granted[dev].load(std::memory_order_acquire) >= bytes) return true;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (granted[dev].load(std::memory_order_relaxed) >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return false;
  granted[dev].store(bytes, std::memory_order_release);
  return true;
}

// First error for a request sticks; kernels never write SPEC_OK.
__device__ __forceinline__ void report(int32_t *status, int b, int code) {
  if (status != nullptr && b >= 0) atomicCAS(status + b, 0, code);
}

// Bounds-checked debug build (-DSPEC_CHECKED): a global access whose index is
// computed from the inputs first asks in_bounds(i, n, ...) whether 0 <= i < n
// for its buffer's extent n.  A failed test records SPEC_ERR_INDEX for request
// b (request 0 when b is not known) and the caller skips the access.  In the
// normal build the test is the constant true and compiles away.
#ifdef SPEC_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

__device__ __forceinline__ bool in_bounds(long long i, long long n, int32_t *status, int b) {
  if constexpr (!kChecked) {
    return true;
  } else {
    if (i >= 0 && i < n) return true;
    report(status, b < 0 ? 0 : b, SPEC_ERR_INDEX);
    return false;
  }
}

// The range [i, i + len) lies inside [0, n).
__device__ __forceinline__ bool range_in_bounds(long long i, long long len, long long n,
                                                int32_t *status, int b) {
  if constexpr (!kChecked) {
    return true;
  } else {
    if (i >= 0 && len >= 0 && i + len <= n) return true;
    report(status, b < 0 ? 0 : b, SPEC_ERR_INDEX);
    return false;
  }
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of phase `parity` (returns at once).
__device__ __forceinline__ bool mbar_poll(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of `bar` to complete; false if `limit_ns` ran out.
// try_wait itself suspends the thread in hardware for a while, so the loop
// polls without sleeping and reads the clock only every 256 polls.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// 4-D tiled bulk-tensor load into this CTA's shared memory, completion
// signalled on `bar` as transaction bytes.  Coordinates are in elements,
// innermost first.
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, uint64_t *bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Bulk copy from this CTA's shared memory to a cluster peer's (`dst` and
// `bar` are shared::cluster addresses in the same peer); completes on the
// peer's barrier.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_s2s(uint32_t dst, uint32_t src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier with release/acquire semantics on shared memory:
// every thread of every CTA in the cluster must execute it.
__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Split cluster barrier: arrive early (relaxed, no ordering), wait later.
// Used once at kernel start so that every CTA of the cluster is known to be
// running before the first access to a peer's shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  __syncwarp();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Address of the same shared-memory object in cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int ld_peer_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_peer_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Remote (distributed shared memory) stores: fire-and-forget, ordered for the
// target CTA by the next cluster barrier.
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_peer_f32x4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// Remote stores that complete on the destination CTA's mbarrier as
// transaction bytes (`addr` and `bar` are shared::cluster addresses of the
// same CTA, from peer_addr).  The destination waits on its barrier; no
// cluster-wide barrier is involved.
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr),
               "f"(v), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_async_v2_f32(uint32_t addr, float x, float y, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::
                   "r"(addr),
               "f"(x), "f"(y), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_async_v4_f32(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

// Named barrier for `nthreads` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %3, 0;\n\t"
      "bar.red.or.pred po, %1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(id), "r"(nthreads), "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0;
}

// 2^x with the hardware approximation (max relative error about 2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x for x <= 127 on the FMA pipe, so that exponential-heavy loops can split
// their work between it and the MUFU pipe (fast_exp2).  Range reduction to
// the nearest integer, x = n + f with |f| <= 1/2, then the degree-7 Taylor
// polynomial of e^(f ln 2) (coefficients (ln 2)^k / k!; truncation error below
// 1e-8 relative on the interval), scaled by 2^n through the exponent field.
// Results below 2^-126 flush to zero, as with ex2.approx.ftz.
__device__ __forceinline__ float exp2_taylor(float x) {
  x = fmaxf(x, -127.f);
  const float n = rintf(x);
  const float f = x - n;
  float p = 1.5252733804059838e-05f;
  p = fmaf(p, f, 1.5403530393381606e-04f);
  p = fmaf(p, f, 1.3333558146428441e-03f);
  p = fmaf(p, f, 9.6181291076284770e-03f);
  p = fmaf(p, f, 5.5504108664821576e-02f);
  p = fmaf(p, f, 2.4022650695910071e-01f);
  p = fmaf(p, f, 6.9314718055994531e-01f);
  p = fmaf(p, f, 1.0f);
  return p * __int_as_float((static_cast<int>(n) + 127) << 23);
}

// ---------------------------------------------------------------- Philox
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11, "Parallel Random Numbers:
// As Easy as 1, 2, 3").  Each round multiplies counter words 0 and 2 by the
// round multipliers, feeds the 128-bit products' halves back with the other
// two words and the round key, and the key advances by the golden-ratio and
// sqrt(3)-derived Weyl increments.
struct U64x4 {
  uint64_t w[4];
};

__device__ __forceinline__ U64x4 philox4x64_10(U64x4 x, uint64_t k0, uint64_t k1) {
  constexpr uint64_t kMul0 = 0xD2E7470EE14C6C93ull;
  constexpr uint64_t kMul1 = 0xCA5A826395121157ull;
  constexpr uint64_t kInc0 = 0x9E3779B97F4A7C15ull;
  constexpr uint64_t kInc1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0_hi = __umul64hi(kMul0, x.w[0]);
    const uint64_t p0_lo = kMul0 * x.w[0];
    const uint64_t p1_hi = __umul64hi(kMul1, x.w[2]);
    const uint64_t p1_lo = kMul1 * x.w[2];
    U64x4 y;
    y.w[0] = p1_hi ^ x.w[1] ^ k0;
    y.w[1] = p1_lo;
    y.w[2] = p0_hi ^ x.w[3] ^ k1;
    y.w[3] = p0_lo;
    x = y;
    k0 += kInc0;
    k1 += kInc1;
  }
  return x;
}

// The method's uniform for (seed, request-local node, request, kind), in
// [0, 1): the top 24 bits of the first output word, exact in fp32.
__device__ __forceinline__ float spec_uniform(uint64_t seed, int node, int request, int kind) {
  U64x4 c;
  c.w[0] = static_cast<uint64_t>(node);
  c.w[1] = static_cast<uint64_t>(request);
  c.w[2] = static_cast<uint64_t>(kind);
  c.w[3] = 0;
  const U64x4 r = philox4x64_10(c, seed, 0);
  return static_cast<float>(r.w[0] >> 40) * (1.0f / 16777216.0f);
}

// Request that owns global node t: the b with off[b] <= t < off[b+1], by
// binary search over monotone offsets.  Returns -1 when none does.
__device__ __forceinline__ int find_request(const int32_t *off, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= t) lo = mid; else hi = mid - 1;
  }
  if (__ldg(off + lo) <= t && t < __ldg(off + lo + 1)) return lo;
  return -1;
}

}  // namespace spec
