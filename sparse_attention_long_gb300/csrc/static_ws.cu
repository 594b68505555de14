// dsa_forward_static_ws: the whole forward without any caller-provided
// workspace.  dsa_forward streams the indexer scores through a ring that the
// caller allocates; this entry point streams them through a fixed ring that
// lives in this library's own device memory instead, so a caller that cannot
// allocate device memory can still run the forward.  Such callers include
// plug-in / custom-operator hosts that hand a library nothing but its input
// and output buffers, and latency-critical loops that must not call
// cudaMalloc (it may synchronise the device) or go through an allocator.
//
// The ring is a file-scope device array of kStaticRingBytes (32 MiB); every
// GPU that loads this library keeps it until the process exits.  Its device
// address is looked up by the first call made with that device current (so
// make that first call before any stream capture), and again only when the
// device's CUDA context has changed since (e.g. after cudaDeviceReset).
// Every call shares the one ring: calls that overlap on the GPU (other
// streams, other host threads) race on it.  The ring needs no clearing: each
// wave's indexer writes every score its top-k then reads.
#include <mutex>

#include "dsa_common.cuh"

namespace dsa {

int ext_check_params(const dsa_params* p, Shape* s);
bool ext_dev_ctx(DevCtx* c);
int ext_attn_fwd_supported(const dsa_params* p, const Shape& s, const void* q, const void* kv,
                           const void* out);
int ext_indexer_rows(const dsa_params* p, const Shape& s, const void* q_I, const void* k_I,
                     const void* w, long long row_begin, long long rows, float* scores,
                     long long ld, DevCtx c, cudaStream_t st);
int ext_attn_fwd(const dsa_params* p, const Shape& s, const void* q, const void* kv,
                 const int32_t* idx, void* out, float* mx, float* sm, DevCtx c, cudaStream_t st);
int launch_topk(const Shape& s, const float* scores, long long ld, long long row_begin,
                long long rows, int32_t* idx, DevCtx c, cudaStream_t st);

CUcontext current_context();

constexpr size_t kStaticRingBytes = 32ull << 20;
static __device__ __align__(256) float g_static_ring[kStaticRingBytes / sizeof(float)];
// device address of g_static_ring per device, with the context it was looked
// up in (looked up again when the current context differs, e.g. after
// cudaDeviceReset reloaded the module)
static std::mutex g_ring_mu;
static CUcontext g_ring_ctx[64];
static float* g_static_ring_addr[64];

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_forward_static_ws(const dsa_params* p, const void* q_I, const void* k_I,
                                     const void* w, const void* q, const void* kv,
                                     int32_t* idx_out, void* out, float* softmax_max,
                                     float* softmax_sum, dsa_stream_t stream) {
  Shape s;
  int rc = ext_check_params(p, &s);
  if (rc) return rc;
  if (!q_I || !k_I || !w || !q || !kv || !idx_out || !out || !softmax_max || !softmax_sum)
    return DSA_ERR_INVALID_ARG;
  if (p->flags & (DSA_FLAG_FP8_INDEXER | DSA_FLAG_FUSED_TOPK)) return DSA_ERR_UNSUPPORTED;  // the ring path only
  rc = ext_attn_fwd_supported(p, s, q, kv, out);
  if (rc) return rc;
  if (p->dtype == DSA_BF16 &&
      ((((uintptr_t)q_I) & 15u) != 0 || (((uintptr_t)k_I) & 15u) != 0))
    return DSA_ERR_INVALID_ARG;
  // rows per wave that fit the fixed ring (a multiple of 4 rows, at least 4)
  const long long total = p->B * p->S_q;
  long long W = (long long)(kStaticRingBytes / (sizeof(float) * (size_t)p->S_k)) / 4 * 4;
  if (W < 4) return DSA_ERR_UNSUPPORTED;  // S_k > 2,097,152: 4 score rows exceed the ring
  if (W > total) W = total;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
  DevCtx c;
  if (!ext_dev_ctx(&c)) return DSA_ERR_CUDA;
  float* ring = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ring_mu);
    CUcontext ctx = current_context();
    if (!ctx || !g_static_ring_addr[dev] || g_ring_ctx[dev] != ctx) {
      float* ptr = nullptr;
      if (cudaGetSymbolAddress((void**)&ptr, g_static_ring) != cudaSuccess || !ptr)
        return DSA_ERR_CUDA;
      ctx = current_context();
      if (!ctx) return DSA_ERR_CUDA;
      g_static_ring_addr[dev] = ptr;
      g_ring_ctx[dev] = ctx;
    }
    ring = g_static_ring_addr[dev];
  }
  cudaStream_t st = (cudaStream_t)stream;
  for (long long r0 = 0; r0 < total; r0 += W) {
    const long long n = (total - r0) < W ? (total - r0) : W;
    rc = ext_indexer_rows(p, s, q_I, k_I, w, r0, n, ring, p->S_k, c, st);
    if (rc) return rc;
    rc = launch_topk(s, ring, p->S_k, r0, n, idx_out + r0 * p->topk, c, st);
    if (rc) return rc;
  }
  return ext_attn_fwd(p, s, q, kv, idx_out, out, softmax_max, softmax_sum, c, st);
}
