// C ABI of the DSA hot path: argument validation, workspace sizing, kernel
// dispatch and the device status word.  See include/dsa.h for the contract.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "dsa_common.cuh"

namespace dsa {

int launch_topk(const Shape& s, const float* scores, long long ld, long long row_begin,
                long long rows, int32_t* idx, DevCtx c, cudaStream_t st);
int launch_simt_indexer(const Shape& s, bool bf16, const void* q_I, const void* k_I, const void* w,
                        long long row_begin, long long rows, float* scores, long long ld, int fill,
                        DevCtx c, cudaStream_t st);
int launch_simt_attn_fwd(const Shape& s, bool bf16, const void* q, const void* kv,
                         const int32_t* idx, void* out, float* mx, float* sm, DevCtx c,
                         cudaStream_t st);
int launch_simt_attn_bwd(const Shape& s, bool bf16, const void* q, const void* kv,
                         const int32_t* idx, const void* out, const void* dout, const float* mx,
                         const float* sm, void* dq, float* dkv, double* ws, DevCtx c,
                         cudaStream_t st);
int launch_simt_kl_bwd(const Shape& s, bool bf16, const void* q, const void* kv, const void* q_I,
                       const void* k_I, const void* w, const int32_t* idx, const float* mx,
                       const float* sm, float* loss, void* dq_I, float* dk_I, float* dw,
                       double* ws, DevCtx c, cudaStream_t st);
size_t simt_smem_attn_fwd(const Shape& s);
size_t simt_smem_attn_bwd(const Shape& s);
size_t simt_smem_kl(const Shape& s);
int launch_quant_e4m3(const void* x, long long nrows, uint8_t* q, float* scale, cudaStream_t st);
int launch_indexer_f8(const Shape& s, const uint8_t* q8, const float* q_scale, const uint8_t* k8,
                      const float* k_scale, const void* w, long long row_begin, long long rows,
                      float* scores, long long ld, DevCtx c, cudaStream_t st);
int launch_indexer_tc(const Shape& s, const void* q_I, const void* k_I, const void* w,
                      long long row_begin, long long rows, float* scores, long long ld, DevCtx c,
                      cudaStream_t st);
int launch_indexer_topk_tc(const Shape& s, const void* q_I, const void* k_I, const void* w,
                           long long row_begin, long long rows, uint32_t* cand_key, int32_t* cand_pos,
                           uint32_t* cand_cnt, long long ld, DevCtx c, cudaStream_t st);
int launch_topk_cand(const Shape& s, const uint32_t* cand_key, const int32_t* cand_pos,
                     const uint32_t* cand_cnt, long long ld, long long row_begin, long long rows,
                     int32_t* idx, DevCtx c, cudaStream_t st);
int launch_attn_fwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx, void* out,
                       float* mx, float* sm, DevCtx c, cudaStream_t st);
size_t bwd_tc_workspace(const Shape& s);
size_t kl_tc_workspace(const Shape& s);
int launch_dsa_bwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx,
                      const void* out, const void* dout, const float* mx, const float* sm,
                      const void* q_I, const void* k_I, const void* w, void* dq, float* dkv,
                      float* loss, void* dq_I, float* dk_I, float* dw, void* ws, DevCtx c,
                      cudaStream_t st);
int launch_attn_bwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx,
                       const void* out, const void* dout, const float* mx, const float* sm,
                       void* dq, float* dkv, void* ws, DevCtx c, cudaStream_t st,
                       float* praw);
int launch_kl_bwd_tc(const Shape& s, const void* q, const void* kv, const void* q_I,
                     const void* k_I, const void* w, const int32_t* idx, const float* mx,
                     const float* sm, float* loss, void* dq_I, float* dk_I, float* dw, void* ws,
                     DevCtx c, cudaStream_t st);

// ------------------------------ status word --------------------------------
// One status word per device (shared by every stream and host thread using
// that device).  Its device address is cached per device together with the
// CUDA context it was looked up in, and looked up again when the current
// context differs (after cudaDeviceReset the module, and the word, are
// reloaded at a new address).
__device__ int g_status;
static unsigned long long g_budget_ns = 2000000000ull;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (CtxGetCurrentFn)p;
  });
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

static std::mutex g_status_mu;
static CUcontext g_status_ctx[64];
static int* g_status_ptr[64];

static bool dev_ctx(DevCtx* c) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(g_status_mu);
  CUcontext ctx = current_context();  // null before the runtime's first call on this thread
  if (!ctx || !g_status_ptr[dev] || g_status_ctx[dev] != ctx) {
    void* p = nullptr;  // (the lookup makes the device's context current if none is)
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess || !p) return false;
    ctx = current_context();
    if (!ctx) return false;
    g_status_ptr[dev] = (int*)p;
    g_status_ctx[dev] = ctx;
  }
  c->status = g_status_ptr[dev];
  c->budget = g_budget_ns;
  return true;
}

// ------------------------------ tensor maps --------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

bool make_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D uint8 tensor map [rows, cols] with a (box_cols x box_rows) box, 128-byte swizzle
bool make_tmap_2d_u8(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                     uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 rows of `ld` floats viewed as [rows][lines][32]: line l of row r holds
// columns [32l, 32l + 32); boxes of box_lines lines with the 128-byte swizzle
bool make_tmap_f32_lines(CUtensorMap* tm, const float* base, uint64_t rows, uint64_t ld,
                         uint64_t lines, uint32_t box_lines) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {32, lines, rows};
  cuuint64_t strides[2] = {128, ld * 4};
  cuuint32_t box[3] = {32, box_lines, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------ validation ---------------------------------
static bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

static bool tc_attn_shape(const dsa_params* p) { return p->H == 128 && p->d_qk == 576 && p->d_v == 512; }
static bool tc_indexer_shape(const dsa_params* p) { return p->H_I == 64 && p->d_I == 128; }

static int check_params(const dsa_params* p, Shape* s) {
  if (!p) return DSA_ERR_INVALID_ARG;
  if (p->layout != DSA_BSND && p->layout != DSA_TND) return DSA_ERR_UNSUPPORTED;
  if (p->cp_mode != DSA_CP_COLOSSAL) return DSA_ERR_UNSUPPORTED;
  if (p->dtype != DSA_BF16 && p->dtype != DSA_FP32) return DSA_ERR_UNSUPPORTED;
  if (p->B < 1 || p->S_q < 1 || p->S_k < 1 || p->H < 1 || p->d_qk < 1 || p->d_v < 1 ||
      p->H_I < 1 || p->d_I < 1 || p->topk < 1)
    return DSA_ERR_INVALID_ARG;
  if (p->layout == DSA_TND && p->B != 1) return DSA_ERR_INVALID_ARG;
  if (p->d_v > p->d_qk) return DSA_ERR_INVALID_ARG;
  if (!(p->scale > 0.f) || !isfinite(p->scale)) return DSA_ERR_INVALID_ARG;
  if (p->S_k > (1ll << 30) || p->S_q > (1ll << 30) || p->B * p->S_q * p->H >= (1ll << 31) ||
      p->B * p->S_k >= (1ll << 31) || p->topk > (1 << 20))
    return DSA_ERR_UNSUPPORTED;
  if (!p->q_row_index && (p->q_row_offset < 0 || p->q_row_offset + p->S_q > p->S_k))
    return DSA_ERR_INVALID_ARG;
  if (p->dtype == DSA_FP32 &&
      (p->H > 1024 || p->d_qk > 1024 || p->H_I > 256 || p->d_I > 512 || p->topk > 8192))
    return DSA_ERR_UNSUPPORTED;
  s->B = (int)p->B;
  s->S_q = (int)p->S_q;
  s->S_k = (int)p->S_k;
  s->H = (int)p->H;
  s->d_qk = (int)p->d_qk;
  s->d_v = (int)p->d_v;
  s->H_I = (int)p->H_I;
  s->d_I = (int)p->d_I;
  s->topk = (int)p->topk;
  s->scale = p->scale;
  s->q_row_offset = p->q_row_offset;
  s->q_row_index = p->q_row_index;
  return DSA_OK;
}

// FP8 indexer operands in the forward's workspace, after the score ring:
// q8 [B*S_q*H_I][128] | k8 [B*S_k][128] | q_scale [B*S_q*H_I] | k_scale [B*S_k],
// each part 256-byte aligned
struct Fp8Buffers {
  size_t q8, k8, sq, sk, total;
};
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
static Fp8Buffers fp8_buffers(const dsa_params* p) {
  Fp8Buffers b;
  const size_t nq = (size_t)(p->B * p->S_q * p->H_I), nk = (size_t)(p->B * p->S_k);
  b.q8 = 0;
  b.k8 = align256(nq * 128);
  b.sq = b.k8 + align256(nk * 128);
  b.sk = b.sq + align256(nq * 4);
  b.total = b.sk + align256(nk * 4);
  return b;
}

static int indexer_rows(const dsa_params* p, const Shape& s, const void* q_I, const void* k_I,
                        const void* w, long long row_begin, long long rows, float* scores,
                        long long ld, bool fill, DevCtx c, cudaStream_t st) {
  const bool bf16 = p->dtype == DSA_BF16;
  if (bf16 && tc_indexer_shape(p)) {
    if (fill) {  // the tensor-core kernel writes causal keys only: pre-fill the rest
      int rc = launch_simt_indexer(s, true, q_I, k_I, w, row_begin, rows, scores, ld, 2, c, st);
      if (rc) return rc;
    }
    return launch_indexer_tc(s, q_I, k_I, w, row_begin, rows, scores, ld, c, st);
  }
  if (bf16 && (size_t)s.H_I * s.d_I * 4 > 96 * 1024) return DSA_ERR_UNSUPPORTED;
  return launch_simt_indexer(s, bf16, q_I, k_I, w, row_begin, rows, scores, ld, fill ? 1 : 0, c, st);
}

static int attn_fwd_supported(const dsa_params* p, const Shape& s, const void* q, const void* kv,
                              const void* out) {
  if (p->dtype == DSA_BF16) {
    if (!tc_attn_shape(p) || p->topk > 2048) return DSA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
  }
  return simt_smem_attn_fwd(s) > 200 * 1024 ? DSA_ERR_UNSUPPORTED : DSA_OK;
}

static int attn_fwd(const dsa_params* p, const Shape& s, const void* q, const void* kv,
                    const int32_t* idx, void* out, float* mx, float* sm, DevCtx c, cudaStream_t st) {
  if (p->dtype == DSA_BF16) return launch_attn_fwd_tc(s, q, kv, idx, out, mx, sm, c, st);
  return launch_simt_attn_fwd(s, false, q, kv, idx, out, mx, sm, c, st);
}

// the tensor-core backward: DeepSeek head shapes, k <= 2048 and a multiple of
// 8 (the [rows*128][k] bf16 intermediates are read by TMA, 16-byte rows)
static bool tc_bwd_shape(const dsa_params* p) {
  return p->dtype == DSA_BF16 && tc_attn_shape(p) && p->topk <= 2048 && p->topk % 8 == 0;
}

// Rows per indexer / top-k wave.  Auto: as many as fit a 256 MB score ring,
// rounded down to a whole number of indexer rounds (4 rows per CTA, one CTA
// per SM), so that no round of a wave runs with idle SMs; when not even one
// round fits (very long rows), 1024 rows.
static long long wave_rows(const dsa_params* p) {
  const long long total = p->B * p->S_q;
  long long w = p->wave_rows;
  if (w <= 0) {
    w = (256ll << 20) / (4 * p->S_k);
    int dev = 0, sms = 0;
    const long long round_rows =
        (cudaGetDevice(&dev) == cudaSuccess &&
         cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
            ? 4ll * sms
            : 1024;
    if (w >= round_rows) w = w / round_rows * round_rows;
    else if (w < 1024) w = 1024;
  }
  w = (w + 3) / 4 * 4;
  return w < total ? w : total;
}

// The fused indexer + top-k: bf16 DeepSeek indexer shapes, S_k < 65536
// (16-bit histogram counts).  Its workspace holds one wave's candidate lists:
// keys [W][S_k] u32 | positions [W][S_k] i32 | counts [W] u32.
static bool fused_topk_shape(const dsa_params* p) {
  return p->dtype == DSA_BF16 && tc_indexer_shape(p) && p->S_k < 65536 &&
         (p->flags & DSA_FLAG_FP8_INDEXER) == 0;
}
static size_t fused_list_bytes(const dsa_params* p) {
  return align256((size_t)wave_rows(p) * (size_t)p->S_k * 4);
}
static size_t fused_topk_workspace(const dsa_params* p) {
  return 2 * fused_list_bytes(p) + align256((size_t)wave_rows(p) * 4);
}
// rows [row_begin, row_begin + rows) in waves of wave_rows
static int indexer_topk_waves(const dsa_params* p, const Shape& s, const void* q_I, const void* k_I,
                              const void* w, long long row_begin, long long rows, int32_t* idx,
                              void* workspace, DevCtx c, cudaStream_t st) {
  const long long W = wave_rows(p);
  uint32_t* ck = (uint32_t*)workspace;
  int32_t* cp = (int32_t*)((uint8_t*)workspace + fused_list_bytes(p));
  uint32_t* cc = (uint32_t*)((uint8_t*)workspace + 2 * fused_list_bytes(p));
  for (long long r0 = row_begin; r0 < row_begin + rows; r0 += W) {
    const long long n = (row_begin + rows - r0) < W ? (row_begin + rows - r0) : W;
    int rc = launch_indexer_topk_tc(s, q_I, k_I, w, r0, n, ck, cp, cc, p->S_k, c, st);
    if (rc) return rc;
    rc = launch_topk_cand(s, ck, cp, cc, p->S_k, r0, n, idx + (r0 - row_begin) * p->topk, c, st);
    if (rc) return rc;
  }
  return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

// bf16 backward in row passes: with 0 < wave_rows < S_q the rows run in
// passes of at most wave_rows rows of one batch, one after the other on the
// stream, and the workspace holds one pass (its P / dS pairs).  Rows are
// independent and dkv, dk_I and the loss accumulate, so the passes give the
// one-pass results (up to the order of the accumulating atomics).
static long long bwd_pass_rows(const dsa_params* p) {
  return (p->wave_rows > 0 && p->wave_rows < p->S_q) ? p->wave_rows : 0;
}
static Shape bwd_ws_shape(const dsa_params* p, const Shape& s) {
  Shape t = s;
  if (const long long W = bwd_pass_rows(p)) {
    t.B = 1;
    t.S_q = (int)W;
  }
  return t;
}
// f(shape, first flattened row, batch) for each pass; one call when unsplit
template <typename F>
static int bwd_passes(const dsa_params* p, const Shape& s, F f) {
  const long long W = bwd_pass_rows(p);
  if (W == 0) return f(s, 0LL, 0LL);
  for (long long b = 0; b < s.B; ++b)
    for (long long r0 = 0; r0 < s.S_q; r0 += W) {
      const long long n = std::min(W, (long long)s.S_q - r0);
      Shape t = s;
      t.B = 1;
      t.S_q = (int)n;
      if (s.q_row_index) t.q_row_index = s.q_row_index + b * s.S_q + r0;
      else t.q_row_offset = s.q_row_offset + r0;
      const int rc = f(t, b * s.S_q + r0, b);
      if (rc) return rc;
    }
  return DSA_OK;
}
template <typename T>
static T* elem_off(T* ptr, long long elems, size_t esz) {
  using B = typename std::conditional<std::is_const<T>::value, const uint8_t, uint8_t>::type;
  return reinterpret_cast<T*>(reinterpret_cast<B*>(ptr) + elems * (long long)esz);
}

extern "C" {

int dsa_version(void) { return 100; }

size_t dsa_workspace_size(const dsa_params* p, int which) {
  Shape s;
  if (check_params(p, &s) != DSA_OK) return 0;
  if (which == DSA_CALL_FORWARD) {
    if (p->flags & DSA_FLAG_FUSED_TOPK) return fused_topk_shape(p) ? fused_topk_workspace(p) : 0;
    size_t bytes = (size_t)wave_rows(p) * (size_t)p->S_k * sizeof(float);
    if (p->flags & DSA_FLAG_FP8_INDEXER) bytes = align256(bytes) + fp8_buffers(p).total;
    return bytes;
  }
  if (which == DSA_CALL_INDEXER_TOPK) return fused_topk_shape(p) ? fused_topk_workspace(p) : 0;
  const Shape sw = bwd_ws_shape(p, s);  // one pass of the bf16 backward
  if (which == DSA_CALL_ATTN_BWD && tc_bwd_shape(p)) return bwd_tc_workspace(sw);
  if (which == DSA_CALL_KL_BWD && tc_bwd_shape(p) && tc_indexer_shape(p)) return kl_tc_workspace(sw);
  if (which == DSA_CALL_BACKWARD) {
    if (tc_bwd_shape(p) && tc_indexer_shape(p)) return bwd_tc_workspace(sw) + kl_tc_workspace(sw);
    const size_t a = dsa_workspace_size(p, DSA_CALL_ATTN_BWD), b = dsa_workspace_size(p, DSA_CALL_KL_BWD);
    return a > b ? a : b;  // the exact path runs the two passes one after the other
  }
  // the exact (fp32) path accumulates dkv / dk_I in fp64 before adding them
  if (which == DSA_CALL_ATTN_BWD && p->dtype == DSA_FP32)
    return (size_t)(p->B * p->S_k * p->d_qk) * sizeof(double);
  if (which == DSA_CALL_KL_BWD && p->dtype == DSA_FP32)
    return (size_t)(p->B * p->S_k * p->d_I) * sizeof(double);
  return 0;
}

int dsa_indexer_scores(const dsa_params* p, const void* q_I, const void* k_I, const void* w,
                       int64_t row_begin, int64_t rows, float* scores, dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!q_I || !k_I || !w || !scores) return DSA_ERR_INVALID_ARG;
  if (row_begin < 0 || rows < 1 || row_begin + rows > p->B * p->S_q) return DSA_ERR_INVALID_ARG;
  if (p->dtype == DSA_BF16 && (!aligned16(q_I) || !aligned16(k_I))) return DSA_ERR_INVALID_ARG;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  const bool fill = (p->flags & DSA_FLAG_CAUSAL_ONLY) == 0;
  return indexer_rows(p, s, q_I, k_I, w, row_begin, rows, scores, p->S_k, fill, c,
                      (cudaStream_t)stream);
}

int dsa_indexer_topk(const dsa_params* p, const void* q_I, const void* k_I, const void* w,
                     int64_t row_begin, int64_t rows, int32_t* idx, void* workspace,
                     dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!fused_topk_shape(p)) return DSA_ERR_UNSUPPORTED;
  if (!q_I || !k_I || !w || !idx) return DSA_ERR_INVALID_ARG;
  if (row_begin < 0 || rows < 1 || row_begin + rows > p->B * p->S_q) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_I) || !aligned16(k_I)) return DSA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  return indexer_topk_waves(p, s, q_I, k_I, w, row_begin, rows, idx, workspace, c,
                            (cudaStream_t)stream);
}

int dsa_indexer_quantize_fp8(const dsa_params* p, const void* q_I, const void* k_I, uint8_t* q8,
                             float* q_scale, uint8_t* k8, float* k_scale, dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (p->dtype != DSA_BF16 || !tc_indexer_shape(p)) return DSA_ERR_UNSUPPORTED;
  if (!q_I || !k_I || !q8 || !q_scale || !k8 || !k_scale) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_I) || !aligned16(k_I) || !aligned16(q8) || !aligned16(k8)) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  rc = launch_quant_e4m3(q_I, p->B * p->S_q * p->H_I, q8, q_scale, st);
  if (rc) return rc;
  return launch_quant_e4m3(k_I, p->B * p->S_k, k8, k_scale, st);
}

int dsa_indexer_scores_fp8(const dsa_params* p, const uint8_t* q8, const float* q_scale,
                           const uint8_t* k8, const float* k_scale, const void* w, int64_t row_begin,
                           int64_t rows, float* scores, dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (p->dtype != DSA_BF16 || !tc_indexer_shape(p)) return DSA_ERR_UNSUPPORTED;
  if (!q8 || !q_scale || !k8 || !k_scale || !w || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8)) return DSA_ERR_INVALID_ARG;
  if (row_begin < 0 || rows < 1 || row_begin + rows > p->B * p->S_q) return DSA_ERR_INVALID_ARG;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  if ((p->flags & DSA_FLAG_CAUSAL_ONLY) == 0) {  // the kernel writes causal keys only: -inf elsewhere
    rc = launch_simt_indexer(s, true, q8, q8, w, row_begin, rows, scores, p->S_k, 2, c, st);
    if (rc) return rc;
  }
  return launch_indexer_f8(s, q8, q_scale, k8, k_scale, w, row_begin, rows, scores, p->S_k, c, st);
}

int dsa_topk(const dsa_params* p, const float* scores, int64_t row_begin, int64_t rows,
             int32_t* idx, dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!scores || !idx) return DSA_ERR_INVALID_ARG;
  if (row_begin < 0 || rows < 1 || row_begin + rows > p->B * p->S_q) return DSA_ERR_INVALID_ARG;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  return launch_topk(s, scores, p->S_k, row_begin, rows, idx, c, (cudaStream_t)stream);
}

int dsa_sparse_attn_fwd(const dsa_params* p, const void* q, const void* kv, const int32_t* idx,
                        void* out, float* softmax_max, float* softmax_sum, void* workspace,
                        dsa_stream_t stream) {
  (void)workspace;
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!q || !kv || !idx || !out || !softmax_max || !softmax_sum) return DSA_ERR_INVALID_ARG;
  rc = attn_fwd_supported(p, s, q, kv, out);
  if (rc) return rc;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  return attn_fwd(p, s, q, kv, idx, out, softmax_max, softmax_sum, c, (cudaStream_t)stream);
}

int dsa_sparse_attn_bwd(const dsa_params* p, const void* q, const void* kv, const int32_t* idx,
                        const void* out, const void* dout, const float* softmax_max,
                        const float* softmax_sum, void* dq, float* dkv, void* workspace,
                        dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!q || !kv || !idx || !out || !dout || !softmax_max || !softmax_sum || !dq || !dkv)
    return DSA_ERR_INVALID_ARG;
  if (tc_bwd_shape(p)) {
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dkv))
      return DSA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
    DevCtx c;
    if (!dev_ctx(&c)) return DSA_ERR_CUDA;
    const long long H = p->H, dqk = p->d_qk, dv = p->d_v, Sk = p->S_k, k = p->topk;
    return bwd_passes(p, s, [&](const Shape& t, long long r, long long b) {
      return launch_attn_bwd_tc(t, elem_off(q, r * H * dqk, 2), elem_off(kv, b * Sk * dqk, 2), idx + r * k,
                                elem_off(out, r * H * dv, 2), elem_off(dout, r * H * dv, 2),
                                softmax_max + r * H, softmax_sum + r * H, elem_off(dq, r * H * dqk, 2),
                                dkv + b * Sk * dqk, workspace, c, (cudaStream_t)stream, nullptr);
    });
  }
  if (p->dtype == DSA_BF16 || simt_smem_attn_bwd(s) > 200 * 1024) return DSA_ERR_UNSUPPORTED;
  if (dsa_workspace_size(p, DSA_CALL_ATTN_BWD) > 0 && !aligned16(workspace)) return DSA_ERR_WORKSPACE;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  return launch_simt_attn_bwd(s, p->dtype == DSA_BF16, q, kv, idx, out, dout, softmax_max,
                              softmax_sum, dq, dkv, (double*)workspace, c, (cudaStream_t)stream);
}

int dsa_indexer_kl_loss_bwd(const dsa_params* p, const void* q, const void* kv, const void* q_I,
                            const void* k_I, const void* w, const int32_t* idx,
                            const float* softmax_max, const float* softmax_sum, float* loss,
                            void* dq_I, float* dk_I, float* dw, void* workspace,
                            dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!q || !kv || !q_I || !k_I || !w || !idx || !softmax_max || !softmax_sum || !loss || !dq_I ||
      !dk_I || !dw)
    return DSA_ERR_INVALID_ARG;
  if (tc_bwd_shape(p) && tc_indexer_shape(p)) {
    if (!aligned16(q) || !aligned16(kv) || !aligned16(k_I) || !aligned16(dk_I) ||
        ((uintptr_t)dq_I & 3u) != 0)
      return DSA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
    DevCtx c;
    if (!dev_ctx(&c)) return DSA_ERR_CUDA;
    const long long H = p->H, dqk = p->d_qk, Sk = p->S_k, k = p->topk, HI = p->H_I, dI = p->d_I;
    return bwd_passes(p, s, [&](const Shape& t, long long r, long long b) {
      return launch_kl_bwd_tc(t, elem_off(q, r * H * dqk, 2), elem_off(kv, b * Sk * dqk, 2),
                              elem_off(q_I, r * HI * dI, 2), elem_off(k_I, b * Sk * dI, 2),
                              elem_off(w, r * HI, 2), idx + r * k, softmax_max + r * H,
                              softmax_sum + r * H, loss, elem_off(dq_I, r * HI * dI, 2),
                              dk_I + b * Sk * dI, dw + r * HI, workspace, c, (cudaStream_t)stream);
    });
  }
  if (p->dtype == DSA_BF16 || simt_smem_kl(s) > 200 * 1024) return DSA_ERR_UNSUPPORTED;
  if (dsa_workspace_size(p, DSA_CALL_KL_BWD) > 0 && !aligned16(workspace)) return DSA_ERR_WORKSPACE;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  return launch_simt_kl_bwd(s, p->dtype == DSA_BF16, q, kv, q_I, k_I, w, idx, softmax_max,
                            softmax_sum, loss, dq_I, dk_I, dw, (double*)workspace, c,
                            (cudaStream_t)stream);
}

int dsa_backward(const dsa_params* p, const void* q, const void* kv, const int32_t* idx,
                 const void* out, const void* dout, const float* softmax_max,
                 const float* softmax_sum, const void* q_I, const void* k_I, const void* w,
                 void* dq, float* dkv, float* loss, void* dq_I, float* dk_I, float* dw,
                 void* workspace, dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!q || !kv || !idx || !out || !dout || !softmax_max || !softmax_sum || !q_I || !k_I || !w ||
      !dq || !dkv || !loss || !dq_I || !dk_I || !dw)
    return DSA_ERR_INVALID_ARG;
  if (tc_bwd_shape(p) && tc_indexer_shape(p)) {
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dkv) || !aligned16(k_I) || !aligned16(dk_I) || ((uintptr_t)dq_I & 3u) != 0)
      return DSA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
    DevCtx c;
    if (!dev_ctx(&c)) return DSA_ERR_CUDA;
    const long long H = p->H, dqk = p->d_qk, dv = p->d_v, Sk = p->S_k, k = p->topk, HI = p->H_I,
                    dI = p->d_I;
    return bwd_passes(p, s, [&](const Shape& t, long long r, long long b) {
      return launch_dsa_bwd_tc(t, elem_off(q, r * H * dqk, 2), elem_off(kv, b * Sk * dqk, 2), idx + r * k,
                               elem_off(out, r * H * dv, 2), elem_off(dout, r * H * dv, 2),
                               softmax_max + r * H, softmax_sum + r * H, elem_off(q_I, r * HI * dI, 2),
                               elem_off(k_I, b * Sk * dI, 2), elem_off(w, r * HI, 2),
                               elem_off(dq, r * H * dqk, 2), dkv + b * Sk * dqk, loss,
                               elem_off(dq_I, r * HI * dI, 2), dk_I + b * Sk * dI, dw + r * HI,
                               workspace, c, (cudaStream_t)stream);
    });
  }
  rc = dsa_sparse_attn_bwd(p, q, kv, idx, out, dout, softmax_max, softmax_sum, dq, dkv, workspace,
                           stream);
  if (rc) return rc;
  return dsa_indexer_kl_loss_bwd(p, q, kv, q_I, k_I, w, idx, softmax_max, softmax_sum, loss, dq_I,
                                 dk_I, dw, workspace, stream);
}

int dsa_forward(const dsa_params* p, const void* q_I, const void* k_I, const void* w,
                const void* q, const void* kv, int32_t* idx_out, void* out, float* softmax_max,
                float* softmax_sum, void* workspace, dsa_stream_t stream) {
  Shape s;
  int rc = check_params(p, &s);
  if (rc) return rc;
  if (!q_I || !k_I || !w || !q || !kv || !idx_out || !out || !softmax_max || !softmax_sum)
    return DSA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
  rc = attn_fwd_supported(p, s, q, kv, out);
  if (rc) return rc;
  if (p->dtype == DSA_BF16 && (!aligned16(q_I) || !aligned16(k_I))) return DSA_ERR_INVALID_ARG;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  const long long total = p->B * p->S_q, W = wave_rows(p);
  if (p->flags & DSA_FLAG_FUSED_TOPK) {
    if (!fused_topk_shape(p)) return DSA_ERR_UNSUPPORTED;
    rc = indexer_topk_waves(p, s, q_I, k_I, w, 0, total, idx_out, workspace, c, st);
    if (rc) return rc;
    return attn_fwd(p, s, q, kv, idx_out, out, softmax_max, softmax_sum, c, st);
  }
  float* ring = (float*)workspace;
  const bool fp8 = (p->flags & DSA_FLAG_FP8_INDEXER) != 0;
  uint8_t *q8 = nullptr, *k8 = nullptr;
  float *sq = nullptr, *sk = nullptr;
  if (fp8) {
    if (p->dtype != DSA_BF16 || !tc_indexer_shape(p)) return DSA_ERR_UNSUPPORTED;
    const Fp8Buffers fb = fp8_buffers(p);
    uint8_t* base = (uint8_t*)workspace + align256((size_t)W * (size_t)p->S_k * sizeof(float));
    q8 = base + fb.q8;
    k8 = base + fb.k8;
    sq = (float*)(base + fb.sq);
    sk = (float*)(base + fb.sk);
    rc = launch_quant_e4m3(q_I, total * p->H_I, q8, sq, st);
    if (rc) return rc;
    rc = launch_quant_e4m3(k_I, p->B * p->S_k, k8, sk, st);
    if (rc) return rc;
  }
  for (long long r0 = 0; r0 < total; r0 += W) {
    const long long n = (total - r0) < W ? (total - r0) : W;
    rc = fp8 ? launch_indexer_f8(s, q8, sq, k8, sk, w, r0, n, ring, p->S_k, c, st)
             : indexer_rows(p, s, q_I, k_I, w, r0, n, ring, p->S_k, false, c, st);
    if (rc) return rc;
    rc = launch_topk(s, ring, p->S_k, r0, n, idx_out + r0 * p->topk, c, st);
    if (rc) return rc;
  }
  return attn_fwd(p, s, q, kv, idx_out, out, softmax_max, softmax_sum, c, st);
}

int dsa_get_status(dsa_stream_t stream, int* device_status) {
  if (!device_status) return DSA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  *device_status = v;
  return DSA_OK;
}

int dsa_set_wait_budget_ns(uint64_t budget_ns) {
  if (budget_ns == 0) return DSA_ERR_INVALID_ARG;
  g_budget_ns = budget_ns;
  return DSA_OK;
}

}  // extern "C"

namespace dsa {
// one warp waits on an mbarrier that nothing completes; the bounded wait gives
// up after the budget and records DSA_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(DevCtx c) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, c, &abort_flag);
}
}  // namespace dsa

extern "C" int dsa_selftest_wait_timeout(uint64_t budget_ns, dsa_stream_t stream) {
  if (budget_ns == 0 || budget_ns > 10000000000ull) return DSA_ERR_INVALID_ARG;
  DevCtx c;
  if (!dev_ctx(&c)) return DSA_ERR_CUDA;
  c.budget = budget_ns;
  selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Thin non-static entry points into the helpers above, for the scratch-free
// forward in static_ws.cu (which adds a separate entry point and reuses these
// unchanged).
namespace dsa {
int ext_check_params(const dsa_params* p, Shape* s) { return check_params(p, s); }
bool ext_dev_ctx(DevCtx* c) { return dev_ctx(c); }
int ext_attn_fwd_supported(const dsa_params* p, const Shape& s, const void* q, const void* kv,
                           const void* out) {
  return attn_fwd_supported(p, s, q, kv, out);
}
int ext_indexer_rows(const dsa_params* p, const Shape& s, const void* q_I, const void* k_I,
                     const void* w, long long row_begin, long long rows, float* scores,
                     long long ld, DevCtx c, cudaStream_t st) {
  return indexer_rows(p, s, q_I, k_I, w, row_begin, rows, scores, ld, false, c, st);
}
int ext_attn_fwd(const dsa_params* p, const Shape& s, const void* q, const void* kv,
                 const int32_t* idx, void* out, float* mx, float* sm, DevCtx c, cudaStream_t st) {
  return attn_fwd(p, s, q, kv, idx, out, mx, sm, c, st);
}
}  // namespace dsa
