// Indexer KL-loss backward on tcgen05 (bf16 in, fp32 accumulate), indexer
// shapes H_I = 64, d_I = 128.
//
// [DSA-32K] SparseLightningIndexerGradKLLoss, per query row t over its
// selected keys:
//   S_j = q_I[t,j] . k_I[idx]          (recomputed on the tensor cores)
//   I   = sum_j w_j ReLU(S_j),  pi = Softmax(I),  p = the attention target
//   loss += sum p (log p - log pi),    dI = pi - p
//   dS_j = dI w_j [S_j > 0],  dw_j = sum dI ReLU(S_j)
//   dq_I[t] = dS K_sel,       dk_I[idx] += dS^T q_I[t]
//
// One CTA per query row, two passes over 128-key tiles:
//   pass A  S^T = K_tile q_I^T (M = 128 keys, N = 64 heads, K = 128) into
//           TMEM; the epilogue (thread = key) forms I.  Then lse, the loss and
//           dI for the row.
//   pass B  S^T again; the epilogue forms dS^T (as a bf16 hi/lo pair, so the
//           two contractions below carry ~16 mantissa bits of dS) and the dw
//           partials; then dk_tile = dS^T q_I (M = 128 keys, N = 128, K = 64)
//           is scattered into dk_I with vector reductions, and
//           dq_I^T += K_tile^T dS^T (M = 128 dims, N = 64 heads, K = 128 keys)
//           accumulates in TMEM across the tiles.
// Warp 0 owns TMEM and issues the MMAs; warps 1..4 gather the key tiles and
// run the epilogues.  Small shared memory and 256 TMEM columns let two CTAs
// share an SM, so one CTA's gathers overlap the other's MMAs.
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace kltc {

constexpr int kHI = 64, kDI = 128, kTile = 128, kMaxK = 2048;
constexpr int kThreads = 160;
constexpr uint32_t kColS = 0, kColDK = 64, kColDQ = 192;   // TMEM columns
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescDK = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdescDQ = idesc_bf16(128, 64, true, true);

struct __align__(1024) Smem {
  uint8_t kt[2][kTile * 128];   // key tile: dims 0..63 | 64..127, [128 keys][128 B] SW128
  uint8_t qi[2][kHI * 128];     // q_I row: dims 0..63 | 64..127, [64 heads][128 B] SW128
  uint8_t ds[2][kTile * 128];   // dS^T hi | lo: [128 keys][64 heads bf16] SW128
  float pv[kMaxK];              // target p per slot
  float iv[kMaxK];              // indexer logit I, then dI
  int32_t idx[kMaxK];
  float wv[kHI];
  float dws[4][kHI];            // per-warp dw partials (summed in a fixed order)
  float red[8];
  uint64_t kt_full, s_done, s_free, ds_full, g_done;
  uint32_t tmem_base;
  int abort;
  int last;
};

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), two values packed as bf16x2
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
  lo = pack_bf16x2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

// sum / max over the 128 worker threads (warps 1..4), result in every worker
__device__ __forceinline__ float workers_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = (threadIdx.x >> 5) - 1;
  named_bar_sync(1, 128);
  if ((threadIdx.x & 31) == 0) red[w] = v;
  named_bar_sync(1, 128);
  return red[0] + red[1] + red[2] + red[3];
}
__device__ __forceinline__ float workers_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = (threadIdx.x >> 5) - 1;
  named_bar_sync(1, 128);
  if ((threadIdx.x & 31) == 0) red[w] = v;
  named_bar_sync(1, 128);
  return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

__global__ void __launch_bounds__(kThreads, 2)
    kl_tc_kernel(Shape s, const __nv_bfloat16* __restrict__ q_I, const __nv_bfloat16* __restrict__ k_I,
                 const __nv_bfloat16* __restrict__ w, const int32_t* __restrict__ idx,
                 const float* __restrict__ praw, float* __restrict__ loss,
                 __nv_bfloat16* __restrict__ dq_I, float* __restrict__ dk_I,
                 float* __restrict__ dw, DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x;
  const long long b = row / s.S_q;
  const int k = s.topk;
  volatile int* abort_flag = &sm.abort;
  const int t = threadIdx.x - 32;                  // worker index 0..127 (warps 1..4)
  const int quad = warp & 3;
  const int my = quad * 32 + lane;                  // TMEM lane of this worker

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.kt_full), 128);
    mbar_init(smem_u32(&sm.s_done), 1);
    mbar_init(smem_u32(&sm.s_free), 128);  // pass A: the workers have read S^T
    mbar_init(smem_u32(&sm.ds_full), 128);
    mbar_init(smem_u32(&sm.g_done), 1);
    sm.abort = 0;
    sm.last = -1;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 256);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  // stage the index row, the target mass and the head weights
  int last = -1;
  for (int i = threadIdx.x; i < k; i += kThreads) {
    int id = idx[row * k + i];
    if (id < 0 || id >= s.S_k) id = -1;
    else last = i;
    sm.idx[i] = id;
    sm.pv[i] = id >= 0 ? praw[row * k + i] : 0.f;
  }
  if (threadIdx.x < kHI) {
    sm.wv[threadIdx.x] = __bfloat162float(w[row * kHI + threadIdx.x]);
  }
  if (last >= 0) atomicMax(&sm.last, last);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int ntile = (sm.last + kTile) / kTile;       // tiles holding a valid slot

  if (warp == 0) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0 && ntile > 0) {
      const uint32_t kt0 = smem_u32(sm.kt[0]), qi0 = smem_u32(sm.qi[0]);
      bool ok = true;
      for (int it = 0; ok && it < 2 * ntile; ++it) {
        ok = mbar_wait(smem_u32(&sm.kt_full), it & 1, c, abort_flag);
        // the previous S^T must have been read before this one overwrites it
        // (in pass B the wait for dS below orders that already)
        if (ok && it >= 1 && it <= ntile)
          ok = mbar_wait(smem_u32(&sm.s_free), (it - 1) & 1, c, abort_flag);
        if (!ok) break;
        fence_proxy_async_smem();  // the gathered key tile (cp.async writes) -> tensor cores
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // S^T = K_tile q_I^T over the 128 dims
          mma_bf16_ss(tmem + kColS, sdesc(kt0 + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024, kSw128),
                      sdesc(qi0 + (kk >> 2) * (kHI * 128) + (kk & 3) * 32, 16, 1024, kSw128), kIdescS,
                      kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&sm.s_done));
        if (it < ntile) continue;
        const int tb = it - ntile;
        ok = mbar_wait(smem_u32(&sm.ds_full), tb & 1, c, abort_flag);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int hl = 0; hl < 2; ++hl) {
          const uint32_t ds0 = smem_u32(sm.ds[hl]);
#pragma unroll
          for (int kh = 0; kh < 4; ++kh)  // dk_tile = dS^T q_I over the 64 heads
            mma_bf16_ss(tmem + kColDK, sdesc(ds0 + kh * 32, 16, 1024, kSw128),
                        sdesc(qi0 + kh * 2048, kHI * 128, 1024, kSw128), kIdescDK,
                        (hl > 0 || kh > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dq^T += K_tile^T dS^T over the 128 keys
            mma_bf16_ss(tmem + kColDQ, sdesc(kt0 + kk * 2048, kTile * 128, 1024, kSw128),
                        sdesc(ds0 + kk * 2048, kTile * 128, 1024, kSw128), kIdescDQ,
                        (tb > 0 || hl > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.g_done));
      }
    }
  } else {
    // --------------------------- workers (thread = key) ---------------------------
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const __nv_bfloat16* kIb = k_I + b * s.S_k * (long long)kDI;
    const uint32_t kt0 = smem_u32(sm.kt[0]);
    bool ok = ntile > 0;
    // q_I row into its swizzled K-major tile (16-byte chunk c of head hh)
    {
      const uint4* src = reinterpret_cast<const uint4*>(q_I + row * (long long)(kHI * kDI));
      const int cch = t & 15;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int hh = (t >> 4) + 8 * i;
        const uint4 v4 = __ldg(src + hh * 16 + cch);
        const uint32_t dst = smem_u32(sm.qi[cch >> 3]) + hh * 128 + (((cch & 7) ^ (hh & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v4.x), "r"(v4.y),
                     "r"(v4.z), "r"(v4.w) : "memory");
      }
    }
    // target p = praw / sum(praw) over the selected keys
    float psum = 0.f;
    for (int i = t; i < k; i += 128) psum += sm.pv[i];
    psum = workers_sum(psum, sm.red);
    const float pinv = psum > 0.f ? 1.f / psum : 0.f;
    for (int i = t; i < k; i += 128) sm.pv[i] *= pinv;
    // k_I rows of the tile's 128 slots, swizzled K-major, copied straight to
    // shared memory (cp.async); kt_full counts each worker's arrive once its
    // copies have landed.  A tile's gather is issued as soon as the key tile
    // is free (the MMAs that read it have completed), so it overlaps the
    // workers' processing of the previous tile.
    auto gather = [&](int tile) {
      const int cch = t & 15;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int key = (t >> 4) + 8 * i;
        const int sl = tile * kTile + key;
        const int id = (sl < k && sm.idx[sl] >= 0) ? sm.idx[sl] : 0;
        cp_async16_cg(kt0 + (cch >> 3) * (kTile * 128) + key * 128 + (((cch & 7) ^ (key & 7)) << 4),
                      reinterpret_cast<const uint4*>(kIb + (long long)id * kDI) + cch);
      }
      cp_async_arrive_noinc(smem_u32(&sm.kt_full));
    };
    auto load_s = [&](uint32_t (&s0)[32], uint32_t (&s1)[32]) {
      tmem_ld32(tmem + lane_off + kColS, s0);
      tmem_ld32(tmem + lane_off + kColS + 32, s1);
      tmem_ld_wait(s0);
      tmem_ld_also(s1);
    };
    int n_s = 0;  // S^T commits consumed so far
    // ---- pass A: indexer logits ----
    if (ok) gather(0);
    for (int tile = 0; ok && tile < ntile; ++tile) {
      ok = mbar_wait_warp(smem_u32(&sm.s_done), n_s & 1, c, abort_flag);
      ++n_s;
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32];
      load_s(s0, s1);
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_free));
      gather(tile + 1 < ntile ? tile + 1 : 0);  // the last one: pass B's first tile
      const int sl = tile * kTile + my;
      float I = -INFINITY;
      if (sl < k && sm.idx[sl] >= 0) {
        I = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          I = fmaf(sm.wv[j], fmaxf(__uint_as_float(s0[j]), 0.f), I);
          I = fmaf(sm.wv[32 + j], fmaxf(__uint_as_float(s1[j]), 0.f), I);
        }
      }
      if (sl < kMaxK) sm.iv[sl] = I;
      tc_fence_before();
    }
    // ---- row statistics: lse, loss, dI ----
    const int nsl = ntile * kTile < k ? ntile * kTile : k;
    named_bar_sync(1, 128);
    float mx = -INFINITY;
    for (int i = t; i < nsl; i += 128) mx = fmaxf(mx, sm.iv[i]);
    mx = workers_max(ok ? mx : -INFINITY, sm.red);
    float es = 0.f;
    if (mx != -INFINITY)
      for (int i = t; i < nsl; i += 128) es += (sm.iv[i] == -INFINITY) ? 0.f : expf(sm.iv[i] - mx);
    es = workers_sum(es, sm.red);
    const float lse = mx + logf(es);
    float lp = 0.f;
    for (int i = t; i < nsl; i += 128) {
      const float I = sm.iv[i], p = sm.pv[i];
      float di = 0.f;
      if (I != -INFINITY) {
        const float logpi = I - lse;
        if (p > 0.f) lp += p * (logf(p) - logpi);
        di = expf(logpi) - p;
      }
      sm.iv[i] = di;
    }
    lp = workers_sum(lp, sm.red);  // also orders the dI writes before pass B reads them
    if (t == 0 && ok && mx != -INFINITY) atomicAdd(loss, lp);
    // ---- pass B: gradients ----
    float dwp[kHI];
#pragma unroll
    for (int j = 0; j < kHI; ++j) dwp[j] = 0.f;
    for (int tile = 0; ok && tile < ntile; ++tile) {
      ok = mbar_wait_warp(smem_u32(&sm.s_done), n_s & 1, c, abort_flag);
      ++n_s;
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32];
      load_s(s0, s1);
      const int sl = tile * kTile + my;
      const bool valid = sl < k && sm.idx[sl] >= 0;
      const float di = valid ? sm.iv[sl] : 0.f;
      // dS^T row of this key (64 heads) as bf16 hi/lo, 8 chunks of 8 heads
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = 8 * ch + 2 * e, j1 = j0 + 1;
          const float S0 = __uint_as_float(j0 < 32 ? s0[j0] : s1[j0 - 32]);
          const float S1 = __uint_as_float(j1 < 32 ? s0[j1] : s1[j1 - 32]);
          const float g0 = S0 > 0.f ? di * sm.wv[j0] : 0.f;
          const float g1 = S1 > 0.f ? di * sm.wv[j1] : 0.f;
          dwp[j0] += S0 > 0.f ? di * S0 : 0.f;
          dwp[j1] += S1 > 0.f ? di * S1 : 0.f;
          split2(g0, g1, hi[e], lo[e]);
        }
        const uint32_t off = my * 128 + ((ch ^ (my & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(sm.ds[0]) + off),
                     "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(sm.ds[1]) + off),
                     "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]) : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.ds_full));
      ok = mbar_wait_warp(smem_u32(&sm.g_done), tile & 1, c, abort_flag);
      if (!ok) break;
      tc_fence_after();
      if (tile + 1 < ntile) gather(tile + 1);  // the key tile is free once dq^T is done
      // scatter this key's dk_I row
      const int id = valid ? sm.idx[sl] : -1;
      float* dst = id < 0 ? nullptr : dk_I + (b * s.S_k + id) * (long long)kDI;
      // this warp's 32 rows of the dS^T hi buffer are its own until it
      // writes the next tile's dS^T (the MMAs that read them are done): they
      // serve as the transpose scratch of the scatter
      const uint32_t scratch = smem_u32(sm.ds[0]) + quad * 4096;
#pragma unroll 1
      for (int cc = 0; cc < kDI; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColDK + cc, v);
        tmem_ld_wait(v);
        warp_scatter_add_32x32(scratch, v, dst == nullptr ? nullptr : dst + cc);
      }
      tc_fence_before();
    }
    cp_async_wait_all();  // no copy may still be in flight when the CTA exits
    // ---- dq_I (thread = dim) and dw ----
    {
      uint32_t q0[32], q1[32];
      const bool have = __all_sync(0xffffffffu, ok);
      if (have) {
        tc_fence_after();
        tmem_ld32(tmem + lane_off + kColDQ, q0);
        tmem_ld32(tmem + lane_off + kColDQ + 32, q1);
        tmem_ld_wait(q0);
        tmem_ld_also(q1);
      }
      __nv_bfloat16* dq = dq_I + row * (long long)(kHI * kDI) + my;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        dq[j * kDI] = __float2bfloat16_rn(have ? __uint_as_float(q0[j]) : 0.f);
        dq[(32 + j) * kDI] = __float2bfloat16_rn(have ? __uint_as_float(q1[j]) : 0.f);
      }
#pragma unroll
      for (int j = 0; j < kHI; ++j) {
        float v = dwp[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sm.dws[warp - 1][j] = v;
      }
      named_bar_sync(1, 128);
      if (t < kHI) dw[row * kHI + t] = ((sm.dws[0][t] + sm.dws[1][t]) + sm.dws[2][t]) + sm.dws[3][t];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace kltc

int launch_kl_tc(const Shape& s, const void* q_I, const void* k_I, const void* w,
                 const int32_t* idx, const float* praw, float* loss, void* dq_I, float* dk_I,
                 float* dw, DevCtx c, cudaStream_t st) {
  using namespace kltc;
  if (s.topk > kMaxK) return DSA_ERR_UNSUPPORTED;
  const size_t smem = sizeof(Smem) + 1024;
  if (cudaFuncSetAttribute(kl_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  const long long rows = (long long)s.B * s.S_q;
  kl_tc_kernel<<<(unsigned)rows, kThreads, smem, st>>>(
      s, (const __nv_bfloat16*)q_I, (const __nv_bfloat16*)k_I, (const __nv_bfloat16*)w, idx, praw,
      loss, (__nv_bfloat16*)dq_I, dk_I, dw, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
