// Sparse multi-query attention forward on tcgen05 (bf16 in, fp32 accumulate).
//
// [DSA-32K] Sparse Flash Attention forward: p[t] = Softmax(q[t] K_topk^T scale),
// O[t] = p[t] V_topk; the 128 heads of token t share its top-k kv rows, each
// row 576 wide (512 latent + 64 rope) and V = its first 512 columns
// (weight-absorbed MLA).
//
// Why a CTA pair per token: one token's O is 128 heads x 512 fp32 = all 512
// TMEM columns of an SM, leaving nothing for the logits.  So the two CTAs of a
// cluster split the columns: CTA c owns V columns [256c, 256c+256) and rope
// columns [512+32c, 512+32c+32) -- 288 of the 576 contraction columns and
// half of O.  Per 64-key block each CTA
//   1. TMA-gathers (tile::gather4) its 288 columns of the 64 selected kv rows,
//   2. computes the partial logits S_c = Q_c K_c^T (M=128 heads, N=64, K=288),
//   3. swaps S_c with its peer through distributed shared memory and forms
//      S = S_0 + S_1 (the same fp32 sum in both CTAs, so both derive the same
//      softmax state and the same P without a second exchange),
//   4. runs the fp32 online softmax (one thread per head, exp2 domain; the
//      running max used for P is only moved when it grows by > 2^8, so the O
//      rescale in TMEM is rare), writes P as bf16 to shared memory,
//   5. accumulates O_c += P V_c (M=128, N=256, K=64) in TMEM; V_c is read from
//      the same gathered tile as an MN-major operand (no second copy).
// No multiply is duplicated across the pair; the only redundant work is the
// exp of the shared logits.
//
// Roles per CTA: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..5 = softmax / exchange / epilogue (thread = head).
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace attn {

constexpr int kH = 128, kDQK = 576, kDV = 512;
constexpr int kBKey = 64;                         // keys per block
constexpr int kStages = 2;
constexpr int kQChunk = kH * 128;                 // 64 cols x 128 heads (SW128)
constexpr int kQRope = kH * 64;                   // 32 cols x 128 heads (SW64)
constexpr int kQBytes = 4 * kQChunk + kQRope;     // 72 KB
constexpr int kKVChunk = kBKey * 128;             // 8 KB
constexpr int kKVRope = kBKey * 64;               // 4 KB
constexpr int kKVStage = 4 * kKVChunk + kKVRope;  // 36 KB
constexpr int kPBytes = kH * 128;                 // 128 heads x 64 keys bf16
constexpr int kXBytes = kH * kBKey * 4;           // 32 KB fp32 partial logits
constexpr int kSoftWarps = 4;
constexpr int kThreads = 64 + kSoftWarps * 32;
constexpr int kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;
constexpr uint32_t kIdescS = idesc_bf16(128, kBKey, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct __align__(1024) Smem {
  uint8_t q[kQBytes];
  uint8_t kv[kStages][kKVStage];
  uint8_t p[2][kPBytes];
  float x[kH * kBKey];
  uint64_t q_full, kv_full[kStages], kv_empty[kStages], s_full[2], s_empty[2], p_full[2],
      p_empty[2], pv_done, x_full, x_free, mma_done;
  uint32_t tmem_base;
  int abort;
  int nblk;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
                       const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kvr,
                       Shape s, const int32_t* __restrict__ idx, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ mx, float* __restrict__ sm_out, long long nrows,
                       DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const long long row = nrows - 1 - (long long)(blockIdx.x >> 1);  // flattened query row
  const long long b = row / s.S_q;
  const int k = s.topk;
  const int32_t* irow = idx + row * (long long)k;
  volatile int* abort_flag = &sm.abort;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.kv_full[i]), 1);
      mbar_init(smem_u32(&sm.kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.s_full[i]), 1);
      mbar_init(smem_u32(&sm.s_empty[i]), kSoftWarps * 32);
      mbar_init(smem_u32(&sm.p_full[i]), kSoftWarps * 32);
      mbar_init(smem_u32(&sm.p_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.pv_done), 1);
    mbar_init(smem_u32(&sm.x_full), kSoftWarps * 32);  // arrivals come from the peer
    mbar_init(smem_u32(&sm.x_free), kSoftWarps * 32);  // arrivals come from the peer
    mbar_init(smem_u32(&sm.mma_done), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // number of 64-slot blocks up to the last valid index of this row
    int last = -1;
    for (int i = lane; i < k; i += 32) {
      const int id = irow[i];
      if (id >= 0 && id < s.S_k) last = i;
      else if (id < -1 || id >= s.S_k) set_status(c, DSA_ERR_INDEX);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (lane == 0) sm.nblk = (last + kBKey) / kBKey;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int nblk = sm.nblk;
  const uint32_t q0 = smem_u32(sm.q);

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (nblk > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_qr);
        tma_prefetch_desc(&tm_kv);
        tma_prefetch_desc(&tm_kvr);
        const uint32_t qb = smem_u32(&sm.q_full);
        mbar_arrive_expect_tx(qb, kQBytes);
        const int qrow = (int)(row * kH);
        for (int i = 0; i < 4; ++i)
          tma_load_2d(q0 + i * kQChunk, &tm_q, (int)(256 * crank + 64 * i), qrow, qb);
        tma_load_2d(q0 + 4 * kQChunk, &tm_qr, (int)(512 + 32 * crank), qrow, qb);
      }
      const int kvbase = (int)(b * s.S_k);
      int j = 0;
      for (; j < nblk; ++j) {
        const int st = j % kStages;
        if (!mbar_wait_warp(smem_u32(&sm.kv_empty[st]), ((j / kStages) & 1) ^ 1, c, abort_flag)) break;
        // this block's 64 rows: lane holds slots lane and lane+32 (invalid -> row 0)
        const int s0 = j * kBKey + lane, s1 = s0 + 32;
        int i0 = s0 < k ? irow[s0] : -1;
        int i1 = s1 < k ? irow[s1] : -1;
        i0 = (i0 >= 0 && i0 < s.S_k) ? kvbase + i0 : kvbase;
        i1 = (i1 >= 0 && i1 < s.S_k) ? kvbase + i1 : kvbase;
        const uint32_t fb = smem_u32(&sm.kv_full[st]);
        const uint32_t dst = smem_u32(sm.kv[st]);
        if (lane == 0) mbar_arrive_expect_tx(fb, kKVStage);
#pragma unroll 1
        for (int g = 0; g < kBKey / 4; ++g) {
          const int src_lane = (g * 4) & 31;
          const int v0 = __shfl_sync(0xffffffffu, g < 8 ? i0 : i1, src_lane + 0);
          const int v1 = __shfl_sync(0xffffffffu, g < 8 ? i0 : i1, src_lane + 1);
          const int v2 = __shfl_sync(0xffffffffu, g < 8 ? i0 : i1, src_lane + 2);
          const int v3 = __shfl_sync(0xffffffffu, g < 8 ? i0 : i1, src_lane + 3);
          if (lane == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              tma_gather4(dst + i * kKVChunk + g * 512, &tm_kv, (int)(256 * crank + 64 * i), v0, v1,
                          v2, v3, fb);
            tma_gather4(dst + 4 * kKVChunk + g * 256, &tm_kvr, (int)(512 + 32 * crank), v0, v1, v2,
                        v3, fb);
          }
        }
      }
      if (lane == 0) {  // drain: every issued copy has landed before exit
        mbar_wait(smem_u32(&sm.q_full), 0, c, abort_flag);
        for (int i = (j > kStages ? j - kStages : 0); i < j; ++i)
          mbar_wait(smem_u32(&sm.kv_full[i % kStages]), (i / kStages) & 1, c, abort_flag);
      }
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0 && nblk > 0) {
      bool ok = mbar_wait(smem_u32(&sm.q_full), 0, c, abort_flag);
      for (int step = 0; ok && step <= nblk; ++step) {
        if (step < nblk) {  // S(step) = Q_c K_c^T
          const int j = step, st = j % kStages, sb = j & 1;
          if (!mbar_wait(smem_u32(&sm.kv_full[st]), (j / kStages) & 1, c, abort_flag)) break;
          if (!mbar_wait(smem_u32(&sm.s_empty[sb]), ((j >> 1) & 1) ^ 1, c, abort_flag)) break;
          tc_fence_after();
          const uint32_t kv0 = smem_u32(sm.kv[st]);
          const uint32_t d = tmem + kColS + sb * kBKey;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            const uint64_t ad = sdesc(q0 + (kk >> 2) * kQChunk + off, 16, 1024, kSw128);
            const uint64_t bd = sdesc(kv0 + (kk >> 2) * kKVChunk + off, 16, 1024, kSw128);
            mma_bf16_ss(d, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t ad = sdesc(q0 + 4 * kQChunk + kk * 32, 16, 512, kSw64);
            const uint64_t bd = sdesc(kv0 + 4 * kKVChunk + kk * 32, 16, 512, kSw64);
            mma_bf16_ss(d, ad, bd, kIdescS, 1u);
          }
          mma_commit(smem_u32(&sm.s_full[sb]));
        }
        if (step >= 1) {  // O_c += P V_c for block step-1
          const int j = step - 1, st = j % kStages, pb = j & 1;
          if (!mbar_wait(smem_u32(&sm.p_full[pb]), (j >> 1) & 1, c, abort_flag)) break;
          tc_fence_after();
          const uint32_t kv0 = smem_u32(sm.kv[st]);
          const uint32_t p0 = smem_u32(sm.p[pb]);
#pragma unroll
          for (int kk = 0; kk < kBKey / 16; ++kk) {
            const uint64_t ad = sdesc(p0 + kk * 32, 16, 1024, kSw128);
            const uint64_t bd = sdesc(kv0 + kk * 2048, kKVChunk, 1024, kSw128);
            mma_bf16_ss(tmem + kColO, ad, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm.kv_empty[st]));
          mma_commit(smem_u32(&sm.p_empty[pb]));
          mma_commit(smem_u32(&sm.pv_done));
        }
      }
      mma_commit(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0, c, abort_flag);
    }
  } else {
    // ----------------------- softmax / exchange / epilogue --------------------
    const int quad = warp & 3;
    const int h = quad * 32 + lane;                      // this thread's head (TMEM lane)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t x_local = smem_u32(sm.x) + h * 256;
    const uint32_t x_remote = mapa_shared(x_local, peer);
    const uint32_t xfull_remote = mapa_shared(smem_u32(&sm.x_full), peer);
    const uint32_t xfree_remote = mapa_shared(smem_u32(&sm.x_free), peer);
    const float sl2e = s.scale * kLog2e;
    float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f, lr_run = 0.f;
    bool ok = true;
    for (int j = 0; ok && j < nblk; ++j) {
      const int sb = j & 1;
      const int s0 = j * kBKey + lane, s1 = s0 + 32;
      const int i0 = s0 < k ? irow[s0] : -1, i1 = s1 < k ? irow[s1] : -1;
      const uint32_t mlo = __ballot_sync(0xffffffffu, i0 >= 0 && i0 < s.S_k);
      const uint32_t mhi = __ballot_sync(0xffffffffu, i1 >= 0 && i1 < s.S_k);
      if (!mbar_wait_warp(smem_u32(&sm.s_full[sb]), (j >> 1) & 1, c, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32(tmem + lane_off + kColS + sb * kBKey, u[0]);
      tmem_ld32(tmem + lane_off + kColS + sb * kBKey + 32, u[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_empty[sb]));
      // send my partial logits to the peer (row h, 16-byte chunks swizzled by h)
      if (!mbar_wait_warp<true>(smem_u32(&sm.x_free), (j & 1) ^ 1, c, abort_flag)) { ok = false; break; }
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint32_t* src = &u[ch >> 3][(ch & 7) * 4];
        st_cluster_v4(x_remote + ((ch ^ (h & 15)) << 4), __uint_as_float(src[0]),
                      __uint_as_float(src[1]), __uint_as_float(src[2]), __uint_as_float(src[3]));
      }
      mbar_arrive_remote(xfull_remote);
      if (!mbar_wait_warp<true>(smem_u32(&sm.x_full), j & 1, c, abort_flag)) { ok = false; break; }
      float v[64];
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const float4 pr = *reinterpret_cast<const float4*>(sm.x + h * 64 + ((ch ^ (h & 15)) << 2));
        const uint32_t* own = &u[ch >> 3][(ch & 7) * 4];
        v[ch * 4 + 0] = __uint_as_float(own[0]) + pr.x;
        v[ch * 4 + 1] = __uint_as_float(own[1]) + pr.y;
        v[ch * 4 + 2] = __uint_as_float(own[2]) + pr.z;
        v[ch * 4 + 3] = __uint_as_float(own[3]) + pr.w;
      }
      mbar_arrive_remote(xfree_remote);
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const bool valid = ((i < 32 ? mlo >> i : mhi >> (i - 32)) & 1u) != 0;
        v[i] = valid ? v[i] * sl2e : -INFINITY;
        bm = fmaxf(bm, v[i]);
      }
      m_true = fmaxf(m_true, bm);
      const bool need = bm > m_run + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = fmaxf(m_run, bm);
        const float alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_new);
        if (j > 0 && __any_sync(0xffffffffu, m_run != -INFINITY)) {
          // O must hold PV(j-1) before it is rescaled
          if (!mbar_wait_warp(smem_u32(&sm.pv_done), (j - 1) & 1, c, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 256; cc += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + kColO + cc, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + lane_off + kColO + cc, o);
          }
          tmem_st_wait();
        }
        l_run *= alpha;
        lr_run *= alpha;
        m_run = m_new;
      }
      const float mu = (m_run == -INFINITY) ? 0.f : m_run;
      if (!mbar_wait_warp(smem_u32(&sm.p_empty[sb]), ((j >> 1) & 1) ^ 1, c, abort_flag)) { ok = false; break; }
      const uint32_t prow = smem_u32(sm.p[sb]) + h * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float pa = ex2(v[ch * 8 + 2 * q] - mu);
          const float pb = ex2(v[ch * 8 + 2 * q + 1] - mu);
          l_run += pa + pb;
          pk[q] = pack_bf16x2(pa, pb);
          __nv_bfloat162 r = *reinterpret_cast<__nv_bfloat162*>(&pk[q]);
          lr_run += __low2float(r) + __high2float(r);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + ((ch ^ (h & 7)) << 4)),
                     "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full[sb]));
    }
    // ------------------------------- epilogue -------------------------------
    bool have = ok && nblk > 0;
    if (have) have = mbar_wait_warp(smem_u32(&sm.pv_done), (nblk - 1) & 1, c, abort_flag);
    tc_fence_after();
    const float inv = (have && lr_run > 0.f) ? 1.f / lr_run : 0.f;
    __nv_bfloat16* orow = out + (row * kH + h) * (long long)kDV + 256 * crank;
#pragma unroll 1
    for (int cc = 0; cc < 256; cc += 32) {
      uint32_t o[32];
      if (__all_sync(0xffffffffu, have)) {
        tmem_ld32(tmem + lane_off + kColO + cc, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      uint4 pk[4];
      uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pw[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
      uint4* dst = reinterpret_cast<uint4*>(orow + cc);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = pk[i];
    }
    if (crank == 0) {
      const bool any = have && m_true != -INFINITY;
      mx[row * kH + h] = any ? m_true * kLn2 : -INFINITY;
      sm_out[row * kH + h] = any ? l_run * ex2(m_run - m_true) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer may still be arriving on our barriers until here
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn

bool make_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

int launch_attn_fwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx, void* out,
                       float* mx, float* sm, DevCtx c, cudaStream_t st) {
  using namespace attn;
  CUtensorMap tq, tqr, tkv, tkvr;
  const uint64_t qrows = (uint64_t)s.B * s.S_q * kH, kvrows = (uint64_t)s.B * s.S_k;
  if (!make_tmap_2d_bf16(&tq, q, qrows, kDQK, 64, kH, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tqr, q, qrows, kDQK, 32, kH, 64)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tkv, kv, kvrows, kDQK, 64, 1, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tkvr, kv, kvrows, kDQK, 32, 1, 64)) return DSA_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  if (cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long nrows = (long long)s.B * s.S_q;
  attn_fwd_tc_kernel<<<(unsigned)(2 * nrows), kThreads, smem, st>>>(
      tq, tqr, tkv, tkvr, s, idx, (__nv_bfloat16*)out, mx, sm, nrows, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
