// CUDA-core (SIMT) kernels for the exact-arithmetic path: fp32 inputs at small
// shapes, fp32 accumulation everywhere.  Tensor cores cannot hold fp32 inputs
// to a 1e-5 agreement, so this path keeps every product in fp32.  Each kernel
// is a direct transcription of one definition, parallel over (row, head).
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {

// [DSA-32K] Lightning Indexer forward: I[t,s] = sum_j w[t,j] ReLU(q_I[t,j].k_I[s]).
// grid (ceil(S_k/128), rows), block 128; one thread per (row, key).
// fill_masked: 0 = causal keys only, 1 = also write -inf for s > pos(t),
// 2 = write only the -inf part (the tensor-core kernel writes the rest).
template <typename T>
__global__ void __launch_bounds__(128)
    simt_indexer_kernel(Shape s, const T* __restrict__ q_I, const T* __restrict__ k_I,
                        const T* __restrict__ w, long long row_begin, float* __restrict__ scores,
                        long long ld, int fill_masked, DevCtx c) {
  extern __shared__ float sh[];
  float* qs = sh;                      // [H_I * d_I]
  float* ws = sh + s.H_I * s.d_I;      // [H_I]
  const long long r_local = blockIdx.y;
  const long long row = row_begin + r_local;
  const long long b = row / s.S_q;
  const long long pos = row_pos(s, row);
  if (fill_masked == 2) {  // only the masked part: s > pos(t) -> -inf
    float* o = scores + r_local * ld;
    const long long key = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (key < s.S_k && (key > pos || pos < 0 || pos >= s.S_k)) o[key] = -INFINITY;
    return;
  }
  const int nq = s.H_I * s.d_I;
  for (int i = threadIdx.x; i < nq; i += blockDim.x) qs[i] = to_f32(q_I[row * nq + i]);
  for (int i = threadIdx.x; i < s.H_I; i += blockDim.x) ws[i] = to_f32(w[row * s.H_I + i]);
  __syncthreads();
  const long long key = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (key >= s.S_k) return;
  float* o = scores + r_local * ld;
  if (pos < 0 || pos >= s.S_k) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(c, DSA_ERR_INDEX);
    if (fill_masked) o[key] = -INFINITY;
    return;
  }
  if (key > pos) {
    if (fill_masked) o[key] = -INFINITY;
    return;
  }
  const T* kr = k_I + (b * s.S_k + key) * s.d_I;
  float acc = 0.f;
  for (int j = 0; j < s.H_I; ++j) {
    const float* qj = qs + j * s.d_I;
    float dot = 0.f;
    for (int d = 0; d < s.d_I; ++d) dot = fmaf(qj[d], to_f32(kr[d]), dot);
    acc = fmaf(ws[j], fmaxf(dot, 0.f), acc);
  }
  o[key] = acc;
}

template <typename T>
__device__ __forceinline__ bool sel_index(const Shape& s, const int32_t* idx_row, int i, int& id,
                                          const DevCtx& c) {
  id = idx_row[i];
  if (id < 0 || id >= s.S_k) {
    if (id < -1 || id >= s.S_k) set_status(c, DSA_ERR_INDEX);
    return false;
  }
  return true;
}

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, y) : v + y;
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < nw; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// [DSA-32K] Sparse Flash Attention forward over the selected rows.
// grid (H, rows), block 128; one CTA per (row, head).
template <typename T>
__global__ void __launch_bounds__(128)
    simt_attn_fwd_kernel(Shape s, const T* __restrict__ q, const T* __restrict__ kv,
                         const int32_t* __restrict__ idx, T* __restrict__ out,
                         float* __restrict__ mx, float* __restrict__ sm_out, DevCtx c) {
  extern __shared__ float sh[];
  float* qh = sh;               // [d_qk]
  float* lg = sh + s.d_qk;      // [topk]
  float* red = lg + s.topk;     // [32]
  const long long row = blockIdx.y;
  const int h = blockIdx.x;
  const long long b = row / s.S_q;
  const int32_t* ir = idx + row * s.topk;
  const T* qr = q + (row * s.H + h) * s.d_qk;
  for (int e = threadIdx.x; e < s.d_qk; e += blockDim.x) qh[e] = to_f32(qr[e]);
  __syncthreads();
  float lmax = -INFINITY;
  for (int i = threadIdx.x; i < s.topk; i += blockDim.x) {
    int id;
    float v = -INFINITY;
    if (sel_index<T>(s, ir, i, id, c)) {
      const T* kr = kv + (b * s.S_k + id) * s.d_qk;
      float dot = 0.f;
      for (int e = 0; e < s.d_qk; ++e) dot = fmaf(qh[e], to_f32(kr[e]), dot);
      v = s.scale * dot;
    }
    lg[i] = v;
    lmax = fmaxf(lmax, v);
  }
  const float m = block_reduce(lmax, red, true);
  T* orow = out + (row * s.H + h) * s.d_v;
  if (m == -INFINITY) {
    for (int e = threadIdx.x; e < s.d_v; e += blockDim.x) orow[e] = from_f32<T>(0.f);
    if (threadIdx.x == 0) {
      mx[row * s.H + h] = -INFINITY;
      sm_out[row * s.H + h] = 0.f;
    }
    return;
  }
  float lsum = 0.f;
  for (int i = threadIdx.x; i < s.topk; i += blockDim.x) {
    const float p = (lg[i] == -INFINITY) ? 0.f : expf(lg[i] - m);
    lg[i] = p;
    lsum += p;
  }
  const float l = block_reduce(lsum, red, false);
  __syncthreads();
  for (int e = threadIdx.x; e < s.d_v; e += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < s.topk; ++i) {
      const int id = ir[i];
      if (id >= 0 && id < s.S_k) acc = fmaf(lg[i], to_f32(kv[(b * s.S_k + id) * s.d_qk + e]), acc);
    }
    orow[e] = from_f32<T>(acc / l);
  }
  if (threadIdx.x == 0) {
    mx[row * s.H + h] = m;
    sm_out[row * s.H + h] = l;
  }
}

// [DSA-32K] SparseFlashAttentionGrad.  grid (H, rows), block 128.
// dkv gets fp32 atomics per (head, key, column): small shapes only.
template <typename T, typename A>
__global__ void __launch_bounds__(128)
    simt_attn_bwd_kernel(Shape s, const T* __restrict__ q, const T* __restrict__ kv,
                         const int32_t* __restrict__ idx, const T* __restrict__ out,
                         const T* __restrict__ dout, const float* __restrict__ mx,
                         const float* __restrict__ sm_in, T* __restrict__ dq,
                         A* __restrict__ dkv, DevCtx c) {
  extern __shared__ float sh[];
  float* qh = sh;                // [d_qk]
  float* dob = qh + s.d_qk;      // [d_v]
  float* P = dob + s.d_v;        // [topk]
  float* dS = P + s.topk;        // [topk]
  float* red = dS + s.topk;      // [32]
  const long long row = blockIdx.y;
  const int h = blockIdx.x;
  const long long b = row / s.S_q;
  const int32_t* ir = idx + row * s.topk;
  const long long rh = row * s.H + h;
  for (int e = threadIdx.x; e < s.d_qk; e += blockDim.x) qh[e] = to_f32(q[rh * s.d_qk + e]);
  float dpart = 0.f;
  for (int e = threadIdx.x; e < s.d_v; e += blockDim.x) {
    const float g = to_f32(dout[rh * s.d_v + e]);
    dob[e] = g;
    dpart = fmaf(g, to_f32(out[rh * s.d_v + e]), dpart);
  }
  const float D = block_reduce(dpart, red, false);  // FlashSoftmaxGrad(dY, O)
  __syncthreads();
  const float m = mx[rh], l = sm_in[rh];
  for (int i = threadIdx.x; i < s.topk; i += blockDim.x) {
    int id;
    float p = 0.f, ds = 0.f;
    if (sel_index<T>(s, ir, i, id, c) && l > 0.f) {
      const T* kr = kv + (b * s.S_k + id) * s.d_qk;
      float dot = 0.f, dp = 0.f;
      for (int e = 0; e < s.d_qk; ++e) dot = fmaf(qh[e], to_f32(kr[e]), dot);
      for (int e = 0; e < s.d_v; ++e) dp = fmaf(dob[e], to_f32(kr[e]), dp);
      p = expf(s.scale * dot - m) / l;
      ds = p * (dp - D);
    }
    P[i] = p;
    dS[i] = ds;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < s.d_qk; e += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < s.topk; ++i) {
      const int id = ir[i];
      if (id >= 0 && id < s.S_k) acc = fmaf(dS[i], to_f32(kv[(b * s.S_k + id) * s.d_qk + e]), acc);
    }
    dq[rh * s.d_qk + e] = from_f32<T>(s.scale * acc);
  }
  for (int i = 0; i < s.topk; ++i) {
    const int id = ir[i];
    if (id < 0 || id >= s.S_k) continue;
    A* dr = dkv + (b * s.S_k + id) * s.d_qk;
    const float gs = s.scale * dS[i], pi = P[i];
    for (int e = threadIdx.x; e < s.d_qk; e += blockDim.x) {
      float v = gs * qh[e];
      if (e < s.d_v) v = fmaf(pi, dob[e], v);
      atomicAdd(dr + e, (A)v);
    }
  }
}

// [DSA-32K] SparseLightningIndexerGradKLLoss.  grid (rows), block 128.
template <typename T, typename A>
__global__ void __launch_bounds__(128)
    simt_kl_bwd_kernel(Shape s, const T* __restrict__ q, const T* __restrict__ kv,
                       const T* __restrict__ q_I, const T* __restrict__ k_I,
                       const T* __restrict__ w, const int32_t* __restrict__ idx,
                       const float* __restrict__ mx, const float* __restrict__ sm_in,
                       float* __restrict__ loss, T* __restrict__ dq_I, A* __restrict__ dk_I,
                       float* __restrict__ dw, DevCtx c) {
  extern __shared__ float sh[];
  float* p = sh;                        // [topk]
  float* I = p + s.topk;                // [topk]
  float* S = I + s.topk;                // [H_I * topk]
  float* qI = S + s.H_I * s.topk;       // [H_I * d_I]
  float* wv = qI + s.H_I * s.d_I;       // [H_I]
  float* red = wv + s.H_I;              // [32]
  const long long row = blockIdx.x;
  const long long b = row / s.S_q;
  const int k = s.topk;
  const int32_t* ir = idx + row * k;
  for (int i = threadIdx.x; i < s.H_I * s.d_I; i += blockDim.x)
    qI[i] = to_f32(q_I[row * s.H_I * s.d_I + i]);
  for (int j = threadIdx.x; j < s.H_I; j += blockDim.x) wv[j] = to_f32(w[row * s.H_I + j]);
  __syncthreads();
  // target p: attention probabilities summed over heads, then L1-normalised
  float psum = 0.f, imax = -INFINITY;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    int id;
    float ph = 0.f, Ii = -INFINITY;
    if (sel_index<T>(s, ir, i, id, c)) {
      const T* kr = kv + (b * s.S_k + id) * s.d_qk;
      for (int h = 0; h < s.H; ++h) {
        const T* qr = q + (row * s.H + h) * s.d_qk;
        float dot = 0.f;
        for (int e = 0; e < s.d_qk; ++e) dot = fmaf(to_f32(qr[e]), to_f32(kr[e]), dot);
        const float l = sm_in[row * s.H + h];
        if (l > 0.f) ph += expf(s.scale * dot - mx[row * s.H + h]) / l;
      }
      const T* kir = k_I + (b * s.S_k + id) * s.d_I;
      Ii = 0.f;
      for (int j = 0; j < s.H_I; ++j) {
        float dot = 0.f;
        for (int d = 0; d < s.d_I; ++d) dot = fmaf(qI[j * s.d_I + d], to_f32(kir[d]), dot);
        S[j * k + i] = dot;
        Ii = fmaf(wv[j], fmaxf(dot, 0.f), Ii);
      }
    } else {
      for (int j = 0; j < s.H_I; ++j) S[j * k + i] = 0.f;
    }
    p[i] = ph;
    I[i] = Ii;
    psum += ph;
    imax = fmaxf(imax, Ii);
  }
  const float P = block_reduce(psum, red, false);
  const float Im = block_reduce(imax, red, true);
  float esum = 0.f;
  for (int i = threadIdx.x; i < k; i += blockDim.x)
    if (I[i] != -INFINITY) esum += expf(I[i] - Im);
  const float lse = Im + logf(block_reduce(esum, red, false));
  float lpart = 0.f;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    float di = 0.f;
    if (I[i] != -INFINITY && P > 0.f) {
      const float pi_ = p[i] / P;
      const float logpi = I[i] - lse;
      if (pi_ > 0.f) lpart += pi_ * (logf(pi_) - logpi);
      di = expf(logpi) - pi_;
    }
    p[i] = di;  // p now holds dI
  }
  const float lt = block_reduce(lpart, red, false);
  if (threadIdx.x == 0 && Im != -INFINITY) atomicAdd(loss, lt);
  __syncthreads();
  for (int j = threadIdx.x; j < s.H_I; j += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < k; ++i) acc = fmaf(p[i], fmaxf(S[j * k + i], 0.f), acc);
    dw[row * s.H_I + j] = acc;
  }
  __syncthreads();  // dw has read S; it is overwritten in place next
  // dS = dI * w * 1[S > 0]  (in place)
  for (int x = threadIdx.x; x < s.H_I * k; x += blockDim.x) {
    const int j = x / k, i = x % k;
    S[x] = (S[x] > 0.f) ? p[i] * wv[j] : 0.f;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < s.H_I * s.d_I; x += blockDim.x) {
    const int j = x / s.d_I, d = x % s.d_I;
    float acc = 0.f;
    for (int i = 0; i < k; ++i) {
      const int id = ir[i];
      if (id >= 0 && id < s.S_k) acc = fmaf(S[j * k + i], to_f32(k_I[(b * s.S_k + id) * s.d_I + d]), acc);
    }
    dq_I[row * s.H_I * s.d_I + x] = from_f32<T>(acc);
  }
  for (int i = 0; i < k; ++i) {
    const int id = ir[i];
    if (id < 0 || id >= s.S_k) continue;
    for (int d = threadIdx.x; d < s.d_I; d += blockDim.x) {
      float acc = 0.f;
      for (int j = 0; j < s.H_I; ++j) acc = fmaf(S[j * k + i], qI[j * s.d_I + d], acc);
      atomicAdd(dk_I + (b * s.S_k + id) * s.d_I + d, (A)acc);
    }
  }
}

// acc[i] += (float)ws[i]: the exact path accumulates atomics in fp64 and adds
// the result into the caller's fp32 accumulator once.
__global__ void add_f64_into_f32(float* __restrict__ acc, const double* __restrict__ ws,
                                 long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    acc[i] += (float)ws[i];
}

// ------------------------------- launchers --------------------------------
template <typename T>
static int launch_simt_indexer_t(const Shape& s, const void* q_I, const void* k_I, const void* w,
                                 long long row_begin, long long rows, float* scores, long long ld,
                                 int fill, DevCtx c, cudaStream_t st) {
  const size_t smem = sizeof(float) * (size_t)(s.H_I * s.d_I + s.H_I);
  dim3 grid((unsigned)((s.S_k + 127) / 128), (unsigned)rows);
  simt_indexer_kernel<T><<<grid, 128, smem, st>>>(s, (const T*)q_I, (const T*)k_I, (const T*)w,
                                                  row_begin, scores, ld, fill, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_simt_indexer(const Shape& s, bool bf16, const void* q_I, const void* k_I, const void* w,
                        long long row_begin, long long rows, float* scores, long long ld, int fill,
                        DevCtx c, cudaStream_t st) {
  return bf16 ? launch_simt_indexer_t<__nv_bfloat16>(s, q_I, k_I, w, row_begin, rows, scores, ld,
                                                     fill, c, st)
              : launch_simt_indexer_t<float>(s, q_I, k_I, w, row_begin, rows, scores, ld, fill, c,
                                             st);
}

size_t simt_smem_attn_fwd(const Shape& s) { return sizeof(float) * (size_t)(s.d_qk + s.topk + 32); }
size_t simt_smem_attn_bwd(const Shape& s) {
  return sizeof(float) * (size_t)(s.d_qk + s.d_v + 2 * s.topk + 32);
}
size_t simt_smem_kl(const Shape& s) {
  return sizeof(float) * (size_t)(2 * s.topk + s.H_I * s.topk + s.H_I * s.d_I + s.H_I + 32);
}

template <typename T, typename K, typename... Args>
static int launch_big_smem(K kernel, dim3 g, size_t smem, cudaStream_t st, Args... args) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return DSA_ERR_CUDA;
  kernel<<<g, 128, smem, st>>>(args...);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_simt_attn_fwd(const Shape& s, bool bf16, const void* q, const void* kv,
                         const int32_t* idx, void* out, float* mx, float* sm, DevCtx c,
                         cudaStream_t st) {
  dim3 g((unsigned)s.H, (unsigned)((long long)s.B * s.S_q));
  const size_t smem = simt_smem_attn_fwd(s);
  if (bf16)
    return launch_big_smem<__nv_bfloat16>(simt_attn_fwd_kernel<__nv_bfloat16>, g, smem, st, s,
                                          (const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx,
                                          (__nv_bfloat16*)out, mx, sm, c);
  return launch_big_smem<float>(simt_attn_fwd_kernel<float>, g, smem, st, s, (const float*)q,
                                (const float*)kv, idx, (float*)out, mx, sm, c);
}

int launch_simt_attn_bwd(const Shape& s, bool bf16, const void* q, const void* kv,
                         const int32_t* idx, const void* out, const void* dout, const float* mx,
                         const float* sm, void* dq, float* dkv, double* ws, DevCtx c,
                         cudaStream_t st) {
  dim3 g((unsigned)s.H, (unsigned)((long long)s.B * s.S_q));
  const size_t smem = simt_smem_attn_bwd(s);
  if (bf16)
    return launch_big_smem<__nv_bfloat16>(
        simt_attn_bwd_kernel<__nv_bfloat16, float>, g, smem, st, s, (const __nv_bfloat16*)q,
        (const __nv_bfloat16*)kv, idx, (const __nv_bfloat16*)out, (const __nv_bfloat16*)dout, mx,
        sm, (__nv_bfloat16*)dq, dkv, c);
  const long long n = (long long)s.B * s.S_k * s.d_qk;
  if (cudaMemsetAsync(ws, 0, sizeof(double) * n, st) != cudaSuccess) return DSA_ERR_CUDA;
  int rc = launch_big_smem<float>(simt_attn_bwd_kernel<float, double>, g, smem, st, s,
                                  (const float*)q, (const float*)kv, idx, (const float*)out,
                                  (const float*)dout, mx, sm, (float*)dq, ws, c);
  if (rc) return rc;
  add_f64_into_f32<<<256, 256, 0, st>>>(dkv, ws, n);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_simt_kl_bwd(const Shape& s, bool bf16, const void* q, const void* kv, const void* q_I,
                       const void* k_I, const void* w, const int32_t* idx, const float* mx,
                       const float* sm, float* loss, void* dq_I, float* dk_I, float* dw,
                       double* ws, DevCtx c, cudaStream_t st) {
  dim3 g((unsigned)((long long)s.B * s.S_q));
  const size_t smem = simt_smem_kl(s);
  if (bf16)
    return launch_big_smem<__nv_bfloat16>(
        simt_kl_bwd_kernel<__nv_bfloat16, float>, g, smem, st, s, (const __nv_bfloat16*)q,
        (const __nv_bfloat16*)kv, (const __nv_bfloat16*)q_I, (const __nv_bfloat16*)k_I,
        (const __nv_bfloat16*)w, idx, mx, sm, loss, (__nv_bfloat16*)dq_I, dk_I, dw, c);
  const long long n = (long long)s.B * s.S_k * s.d_I;
  if (cudaMemsetAsync(ws, 0, sizeof(double) * n, st) != cudaSuccess) return DSA_ERR_CUDA;
  int rc = launch_big_smem<float>(simt_kl_bwd_kernel<float, double>, g, smem, st, s,
                                  (const float*)q, (const float*)kv, (const float*)q_I,
                                  (const float*)k_I, (const float*)w, idx, mx, sm, loss,
                                  (float*)dq_I, ws, dw, c);
  if (rc) return rc;
  add_f64_into_f32<<<256, 256, 0, st>>>(dk_I, ws, n);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
