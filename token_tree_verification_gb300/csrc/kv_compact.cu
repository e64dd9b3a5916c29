// The depth-first KV-cache update after verification.
//
// SpecInfer news write-up, "Token 樹驗證器": the verifier's KV cache is
// updated depth-first, so the accepted path becomes the next step's prefix
// without extra storage.  Slot L + j receives the old slot L + path[j]
// (j = 1 .. acc) in the K and V caches of every KV head.
//
// One CTA per (KV head, request): every accepted row of K and V is read into
// shared memory first and written back after one barrier (a destination slot
// may be the source of a later path entry), in 16-byte chunks.
#include "common.cuh"

namespace spec {

namespace {

constexpr int kKvThreads = 256;

struct KvArgs {
  uint8_t *k, *v;
  int es, B, H, D, S_cap, W;
  const int32_t *prefix, *offsets, *path, *accept;
  int32_t *new_prefix, *status;
};

__global__ void __launch_bounds__(kKvThreads)
kv_compact_kernel(const KvArgs a) {
  extern __shared__ __align__(16) uint4 rows[];   // [2][acc][row chunks]
  __shared__ int s_ok, s_acc, s_L;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  if (tid == 0) {
    const int L = __ldg(a.prefix + b);
    int ok = __ldcg(a.status + b) == 0;
    int acc = 0;
    if (ok) {
      const int n = __ldg(a.offsets + b + 1) - __ldg(a.offsets + b);
      acc = __ldg(a.accept + b);
      const int32_t *pn = a.path + static_cast<size_t>(b) * a.W;
      int err = 0;
      if (L < 0 || L + n > a.S_cap) {
        err = SPEC_ERR_PREFIX_RANGE;
      } else if (acc < 0 || acc + 1 > a.W) {
        err = SPEC_ERR_TREE_TOO_LARGE;
      } else {
        int prev = __ldg(pn);
        if (prev != 0) err = SPEC_ERR_BAD_PARENT;
        for (int j = 1; j <= acc && !err; ++j) {
          const int x = __ldg(pn + j);
          if (x <= prev || x >= n) err = SPEC_ERR_BAD_PARENT;
          prev = x;
        }
      }
      if (err) {
        if (h == 0) report(a.status, b, err);
        ok = 0;
      }
    }
    if (h == 0) a.new_prefix[b] = ok ? L + 1 + acc : L;
    s_ok = ok;
    s_acc = ok ? acc : 0;
    s_L = L;
  }
  __syncthreads();
  const int acc = s_acc;
  if (!s_ok || acc == 0) return;
  const int L = s_L;
  const int32_t *pn = a.path + static_cast<size_t>(b) * a.W;
  const int chunks = a.D * a.es / 16;                 // 16-byte chunks per row
  const size_t row_bytes = static_cast<size_t>(a.D) * a.es;
  const size_t head = (static_cast<size_t>(b) * a.H + h) * a.S_cap;
  const int total = 2 * acc * chunks;
  for (int i = tid; i < total; i += kKvThreads) {
    const int kv = i / (acc * chunks), rem = i % (acc * chunks);
    const int j = rem / chunks, c = rem % chunks;
    const int x = __ldg(pn + j + 1);
    const uint8_t *src = (kv ? a.v : a.k) + (head + L + x) * row_bytes;
    rows[i] = in_bounds(L + x, a.S_cap, a.status, b) ? __ldcs(reinterpret_cast<const uint4 *>(src) + c)
                                                      : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  for (int i = tid; i < total; i += kKvThreads) {
    const int kv = i / (acc * chunks), rem = i % (acc * chunks);
    const int j = rem / chunks, c = rem % chunks;
    uint8_t *dst = (kv ? a.v : a.k) + (head + L + 1 + j) * row_bytes;
    if (in_bounds(L + 1 + j, a.S_cap, a.status, b)) reinterpret_cast<uint4 *>(dst)[c] = rows[i];
  }
}

}  // namespace

}  // namespace spec

extern "C" int spec_kv_compact(void *k_cache, void *v_cache, int dtype, int B, int Hkv, int D,
                               int S_cap, const int32_t *prefix_lens,
                               const int32_t *tree_offsets, const int32_t *path_nodes,
                               const int32_t *accept_len, int max_depth_plus1,
                               int32_t *new_prefix_lens, int32_t *status, void *stream) {
  using namespace spec;
  if (!k_cache || !v_cache || !prefix_lens || !tree_offsets || !path_nodes || !accept_len ||
      !new_prefix_lens || !status)
    return SPEC_ERR_NULL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  const int es = dtype == SPEC_F32 ? 4 : 2;
  if (B < 1 || Hkv < 1 || S_cap < 1 || max_depth_plus1 < 1 || max_depth_plus1 > SPEC_MAX_TREE_NODES ||
      D < 8 || (D * es) % 16 != 0 || B > 65535)
    return SPEC_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(k_cache) & 15) || (reinterpret_cast<uintptr_t>(v_cache) & 15))
    return SPEC_ERR_ALIGNMENT;
  KvArgs args;
  args.k = static_cast<uint8_t *>(k_cache);
  args.v = static_cast<uint8_t *>(v_cache);
  args.es = es;
  args.B = B;
  args.H = Hkv;
  args.D = D;
  args.S_cap = S_cap;
  args.W = max_depth_plus1;
  args.prefix = prefix_lens;
  args.offsets = tree_offsets;
  args.path = path_nodes;
  args.accept = accept_len;
  args.new_prefix = new_prefix_lens;
  args.status = status;
  // room for every row an accepted path can move (acc <= max_depth_plus1 - 1)
  const size_t smem = static_cast<size_t>(2) * (max_depth_plus1 - 1) * D * es;
  if (smem > 200 * 1024) return SPEC_ERR_SHAPE;
  static std::atomic<size_t> granted[kMaxDevices];
  if (smem > 48 * 1024 && !allow_dynamic_smem(kv_compact_kernel, smem, granted)) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(Hkv), static_cast<unsigned>(B), 1);
  cfg.blockDim = dim3(kKvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  pdl_attribute(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_compact_kernel, args) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
