// Backward of the sparse attention and the target side of the indexer KL loss
// on tcgen05 (bf16 in, fp32 accumulate), DeepSeek-V3.2 shapes (128 heads,
// d_qk 576, d_v 512).
//
// [DSA-32K] SparseFlashAttentionGrad: gather K_topk, recompute P, dP = dY V^T,
// dS = P * (dP - FlashSoftmaxGrad(dY, O)), dQ = dS K_topk / sqrt(d),
// dK = ScatterAdd(dS^T Q / sqrt(d)), dV = P^T dY.
//
// A token's operands (q 128x576, dO 128x512) and its accumulators (dQ
// 128x576, a key block's dKV slice) do not fit one SM's shared or tensor
// memory together, so the backward is split into GEMM-shaped passes with the
// per-pair intermediates materialised in HBM (bf16, [rows][128][k]):
//   rowdot  D[t,h]  = sum_e dO*O                                  (SIMT)
//   scores  S, dP   per (token, 128-key tile) in TMEM; epilogue writes
//           P = exp(scale*S - m)/l and scale*dS = scale*P*(dP - D)
//   dq      dQ[t]   = (scale*dS) K_sel           per (token, 192-col tile)
//   dkv     dKV_sel += (scale*dS)^T Q + P^T dO   per (token, col tile), all key
//           tiles, persistent; scattered with fp32 vector reductions.
// The same scores kernel in its logits-only form gives the head-summed
// attention probabilities the indexer KL loss needs (kl_tc.cu takes it from
// there).
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace bwd {

constexpr int kH = 128, kDQK = 576, kDV = 512;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------- rowdot ------------------------------------
// One warp per (row, head): D = sum over the 512 value columns of dO * O.
__global__ void rowdot_kernel(const __nv_bfloat16* __restrict__ dout,
                              const __nv_bfloat16* __restrict__ out, float* __restrict__ D,
                              long long nrh) {
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= nrh) return;
  const uint4* a = reinterpret_cast<const uint4*>(dout + w * kDV);
  const uint4* b = reinterpret_cast<const uint4*>(out + w * kDV);
  float acc = 0.f;
#pragma unroll
  for (int i = lane; i < kDV / 8; i += 32) {
    const uint4 x = a[i], y = b[i];
    const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* yp = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 xf = __bfloat1622float2(xp[q]), yf = __bfloat1622float2(yp[q]);
      acc = fmaf(xf.x, yf.x, fmaf(xf.y, yf.y, acc));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) D[w] = acc;
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), for two values packed
// as bf16x2 (first value in the low half)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
  lo = pack_bf16x2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

// ------------------------------- scores ------------------------------------
// CTA = (row, 128-key tile).  The contraction runs over 9 column chunks of 64
// (8 latent + rope) through a 2-stage ring; stage i holds the tile's kv chunk
// i (gathered), q chunk i and, for the gradient, dO chunk i (TMA), so chunk i
// of kv serves both S and dP before its stage is released.  ~97 KB of shared
// memory and 256 TMEM columns let two CTAs share an SM.  warp 0: TMEM + MMA;
// warp 1: TMA of the q / dO chunks; warps 2..5: gather the kv chunks, then the
// epilogue (thread = head).
constexpr int kSTile = 128;
constexpr int kSThreads = 192;
constexpr int kSStages = 2;
constexpr int kSChunk = kSTile * 128;            // 16 KB: 128 rows x 64 columns
struct __align__(1024) ScoresSmem {
  uint8_t st[kSStages][3][kSChunk];  // [stage][kv | q | dO]; reused as a [128 keys][129] fp32 buffer
  int32_t idx[kSTile];
  uint32_t mask[kSTile / 32];
  uint64_t full[kSStages], empty[kSStages], done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(ScoresSmem) >= kSTile * (kH + 1) * 4, "transpose buffer");

template <bool kGrad>
__global__ void __launch_bounds__(kSThreads, 2)
    scores_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __nv_bfloat16* __restrict__ kv, Shape s, const int32_t* __restrict__ idx,
                  const float* __restrict__ mx, const float* __restrict__ lsum,
                  const float* __restrict__ Dg, __nv_bfloat16* __restrict__ P_ws,
                  __nv_bfloat16* __restrict__ Plo_ws, __nv_bfloat16* __restrict__ dS_ws,
                  __nv_bfloat16* __restrict__ dSlo_ws,
                  float* __restrict__ praw, int ntile,
                  DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  ScoresSmem& sm = *reinterpret_cast<ScoresSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x / ntile;
  const int tile = blockIdx.x % ntile;
  const long long b = row / s.S_q;
  const int k = s.topk;
  const int slot0 = tile * kSTile;
  volatile int* abort_flag = &sm.abort;
  constexpr int nC = 9;  // column chunks: 8 latent (S and dP) + 1 rope (S only)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSStages; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1 + 128);  // TMA arrive (+ bytes) and the gatherers
      mbar_init(smem_u32(&sm.empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.done), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < kSTile) {
    const int sl = slot0 + threadIdx.x;
    int id = sl < k ? idx[row * k + sl] : -1;
    if (id < -1 || id >= s.S_k) set_status(c, DSA_ERR_INDEX);
    if (id < 0 || id >= s.S_k) id = -1;
    sm.idx[threadIdx.x] = id;
    const uint32_t bal = __ballot_sync(0xffffffffu, id >= 0);
    if (lane == 0) sm.mask[threadIdx.x >> 5] = bal;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 256);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const bool any = (sm.mask[0] | sm.mask[1] | sm.mask[2] | sm.mask[3]) != 0u;

  if (any) {
    if (warp == 1) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        if (kGrad) tma_prefetch_desc(&tm_do);
        const int y = (int)(row * kH);
        for (int i = 0; i < nC; ++i) {
          const int st = i % kSStages;
          if (!mbar_wait(smem_u32(&sm.empty[st]), ((i / kSStages) & 1) ^ 1, c, abort_flag)) break;
          const uint32_t fb = smem_u32(&sm.full[st]);
          const bool with_do = kGrad && i < 8;
          mbar_arrive_expect_tx(fb, (with_do ? 2 : 1) * kSChunk);
          tma_load_2d(smem_u32(sm.st[st][1]), &tm_q, 64 * i, y, fb);
          if (with_do) tma_load_2d(smem_u32(sm.st[st][2]), &tm_do, 64 * i, y, fb);
        }
        for (int i = nC - kSStages; i < nC; ++i)  // drain: no copy left in flight
          mbar_wait(smem_u32(&sm.full[i % kSStages]), (i / kSStages) & 1, c, abort_flag);
      }
    } else if (warp >= 2) {
      // gather chunk i of the tile's 128 kv rows: thread = (key, 16-byte piece)
      const int t = threadIdx.x - 64;
      const int cc = t & 7;
      const __nv_bfloat16* kvb = kv + b * s.S_k * (long long)kDQK;
      for (int i = 0; i < nC; ++i) {
        const int st = i % kSStages;
        if (!mbar_wait_warp(smem_u32(&sm.empty[st]), ((i / kSStages) & 1) ^ 1, c, abort_flag)) break;
        // straight into the swizzled stage (cp.async): the next chunks are
        // issued while this one is in flight; full[st] counts this thread's
        // arrive once its copies have landed, and the MMA issuer fences them
        // into the async proxy
        const uint32_t kvs = smem_u32(sm.st[st][0]);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int key = (t >> 3) + 16 * m;
          const int id = sm.idx[key] < 0 ? 0 : sm.idx[key];
          cp_async16_cg(kvs + key * 128 + ((cc ^ (key & 7)) << 4),
                        reinterpret_cast<const uint4*>(kvb + (long long)id * kDQK + 64 * i) + cc);
        }
        cp_async_arrive_noinc(smem_u32(&sm.full[st]));
      }
      cp_async_wait_all();  // no copy may still be in flight when the CTA exits
    } else if (lane == 0) {
      // MMA: S (TMEM cols 0..127) and dP (cols 128..255), M=128 heads, N=128 keys
      constexpr uint32_t idesc = idesc_bf16(128, kSTile, false, false);
      bool ok = true;
      for (int i = 0; ok && i < nC; ++i) {
        const int st = i % kSStages;
        ok = mbar_wait(smem_u32(&sm.full[st]), (i / kSStages) & 1, c, abort_flag);
        if (!ok) break;
        fence_proxy_async_smem();  // the gathered kv chunk (cp.async writes) -> tensor cores
        tc_fence_after();
        const uint32_t kv0 = smem_u32(sm.st[st][0]), q0 = smem_u32(sm.st[st][1]),
                       o0 = smem_u32(sm.st[st][2]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tmem, sdesc(q0 + kk * 32, 16, 1024, kSw128),
                      sdesc(kv0 + kk * 32, 16, 1024, kSw128), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        if (kGrad && i < 8) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(tmem + 128, sdesc(o0 + kk * 32, 16, 1024, kSw128),
                        sdesc(kv0 + kk * 32, 16, 1024, kSw128), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.empty[st]));
      }
      mma_commit(smem_u32(&sm.done));
    }
  }
  if (warp >= 2) {
    // --------------------------- epilogue: thread = head ---------------------------
    const int quad = warp & 3;
    const int h = quad * 32 + lane;
    const long long rh = row * kH + h;
    bool have = any && mbar_wait_warp(smem_u32(&sm.done), 0, c, abort_flag);
    tc_fence_after();
    const float mh = mx[rh] * kLog2e;
    const float lv = lsum[rh];
    const float linv = lv > 0.f ? 1.f / lv : 0.f;
    const float sl2e = s.scale * kLog2e;
    const float Dh = kGrad ? Dg[rh] : 0.f;
    // The ring is free once the MMAs are done: it stages each 32-key chunk of
    // the four bf16 outputs ([array][head][32 keys], 80-byte row pitch) so the
    // global stores go out as whole 64-byte row segments, and keeps the
    // per-warp head sums of P ([quadrant][key]) for the KL target.
    constexpr int kPitch = 80;
    uint8_t* stg = &sm.st[0][0][0];
    float* psum = reinterpret_cast<float*>(stg + 4 * kH * kPitch);
    const bool colsum = !kGrad || praw != nullptr;
    const int t = threadIdx.x - 64;
#pragma unroll 1
    for (int cc = 0; cc < kSTile; cc += 32) {
      uint32_t sv[32], dv[32];
      if (have) {
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + cc, sv);
        if (kGrad) tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + 128 + cc, dv);
        tmem_ld_wait(sv);
        if (kGrad) tmem_ld_also(dv);
      }
      const uint32_t vm = sm.mask[cc >> 5];
      float p[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        p[i] = (have && ((vm >> i) & 1u)) ? ex2(fmaf(__uint_as_float(sv[i]), sl2e, -mh)) * linv : 0.f;
      if (kGrad) {
        // P and scale*dS as bf16 pairs hi + lo, hi = bf16(x), lo = bf16(x - hi):
        // the later passes contract both halves, so the products carry ~16
        // mantissa bits of P and dS instead of 8
        uint32_t pk[4][16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float d0 = have ? p[2 * i] * (__uint_as_float(dv[2 * i]) - Dh) * s.scale : 0.f;
          const float d1 = have ? p[2 * i + 1] * (__uint_as_float(dv[2 * i + 1]) - Dh) * s.scale : 0.f;
          split_bf16x2(p[2 * i], p[2 * i + 1], pk[0][i], pk[1][i]);
          split_bf16x2(d0, d1, pk[2][i], pk[3][i]);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             smem_u32(stg + (a * kH + h) * kPitch + 16 * i)),
                         "r"(pk[a][4 * i]), "r"(pk[a][4 * i + 1]), "r"(pk[a][4 * i + 2]),
                         "r"(pk[a][4 * i + 3]) : "memory");
      }
      if (colsum) {
        // sum p over this warp's 32 heads for each of the 32 keys (recursive
        // halving: lane L ends with key L's sum), in a fixed order
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < o; ++i) {
            const float send = up ? p[i] : p[i + o];
            const float keep = up ? p[i + o] : p[i];
            p[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        psum[quad * kSTile + cc + lane] = p[0];
      }
      if (kGrad) {
        named_bar_sync(1, 128);  // the chunk is staged
        const int piece = t & 3;
#pragma unroll
        for (int r = 0; r < 16; ++r) {  // 4 arrays x 128 rows x 4 pieces of 16 bytes
          const int a = r >> 2, hh = ((t >> 2) + 32 * r) & 127;
          __nv_bfloat16* arr = a == 0 ? P_ws : a == 1 ? Plo_ws : a == 2 ? dS_ws : dSlo_ws;
          if (slot0 + cc + 8 * piece < k) {  // k is a multiple of 8
            const uint4 v4 = *reinterpret_cast<const uint4*>(stg + (a * kH + hh) * kPitch + 16 * piece);
            *reinterpret_cast<uint4*>(arr + (row * kH + hh) * (long long)k + slot0 + cc + 8 * piece) = v4;
          }
        }
        named_bar_sync(1, 128);  // before the next chunk overwrites the staging
      }
    }
    if (colsum) {
      named_bar_sync(1, 128);
      const int key = t;  // thread = key: the four quadrants' sums in a fixed order
      const float acc = ((psum[key] + psum[kSTile + key]) + psum[2 * kSTile + key]) + psum[3 * kSTile + key];
      if (slot0 + key < k) praw[row * k + slot0 + key] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// --------------------------------- dq ---------------------------------------
// CTA = (row, column tile of dQ: [0, 320) or [320, 576)).  dQ[t, :, cols] =
// sum over key chunks of (scale*dS)[128 heads x 64 keys] * K_sel[64 keys x
// cols], with scale*dS taken as its bf16 pair hi + lo (two MMAs per chunk on
// the same K tile: N = 256 + 64 or N = 256).  Two tiles per row (rather than
// three of 192 columns) read each row's dS chunks twice instead of three
// times.  warp 0: MMA; warp 1: TMA of the dS chunks; warps 2..5: gather the
// 64 kv rows' columns (MN-major SW128: 5 or 4 atoms of 64 columns), then the
// epilogue.
constexpr int kQStages = 3;
constexpr int kQAtoms = 5;              // 64-column atoms of the wider column tile
constexpr int kQSplit = 320;            // column tiles [0, 320) and [320, 576)
struct __align__(1024) DqSmem {
  uint8_t a[kQStages][2][kH * 128];     // dS hi, lo chunks: 128 heads x 64 keys, K-major
  uint8_t bm[kQStages][kQAtoms * 64 * 128];  // 64 keys x up to 320 cols, MN-major
  int32_t idx[2048];
  uint64_t full[kQStages], empty[kQStages], done;
  uint32_t tmem_base;
  int abort;
  int last;
};
static_assert(sizeof(DqSmem) + 1024 <= 232448, "dq shared memory");

__global__ void __launch_bounds__(192, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_dslo,
              const __nv_bfloat16* __restrict__ kv,
              Shape s, const int32_t* __restrict__ idx, __nv_bfloat16* __restrict__ dq, DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem& sm = *reinterpret_cast<DqSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x / 2;
  const int nt = blockIdx.x % 2;
  const int col0 = nt == 0 ? 0 : kQSplit;
  const int natoms = nt == 0 ? kQAtoms : (kDQK - kQSplit) / 64;  // 5 | 4
  const long long b = row / s.S_q;
  const int k = s.topk;
  volatile int* abort_flag = &sm.abort;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1 + 128);
      mbar_init(smem_u32(&sm.empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.done), 1);
    sm.abort = 0;
    sm.last = -1;
    fence_mbar_init();
  }
  __syncthreads();
  int last = -1;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    int id = idx[row * k + i];
    if (id < 0 || id >= s.S_k) id = -1;
    else last = i;
    sm.idx[i] = id;
  }
  if (last >= 0) atomicMax(&sm.last, last);
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);  // 320 columns used
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int nch = (sm.last + 64) / 64;

  if (warp == 1) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_ds);
      tma_prefetch_desc(&tm_dslo);
      for (int ch = 0; ch < nch; ++ch) {
        const int st = ch % kQStages;
        if (!mbar_wait(smem_u32(&sm.empty[st]), ((ch / kQStages) & 1) ^ 1, c, abort_flag)) break;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, 2 * kH * 128);
        tma_load_2d(smem_u32(sm.a[st][0]), &tm_ds, 64 * ch, (int)(row * kH), fb);
        tma_load_2d(smem_u32(sm.a[st][1]), &tm_dslo, 64 * ch, (int)(row * kH), fb);
      }
      for (int ch = (nch > kQStages ? nch - kQStages : 0); ch < nch; ++ch)
        mbar_wait(smem_u32(&sm.full[ch % kQStages]), (ch / kQStages) & 1, c, abort_flag);
    }
  } else if (warp >= 2) {
    const int gw = warp - 2;
    const __nv_bfloat16* kvb = kv + b * s.S_k * (long long)kDQK + col0;
    for (int ch = 0; ch < nch; ++ch) {
      const int st = ch % kQStages;
      if (!mbar_wait_warp(smem_u32(&sm.empty[st]), ((ch / kQStages) & 1) ^ 1, c, abort_flag)) break;
      // straight into the swizzled stage (cp.async), as in the scores kernel
      const uint32_t bs = smem_u32(sm.bm[st]);
      for (int pc = lane; pc < natoms * 8; pc += 32) {  // 16-byte piece pc of the tile's row
        const int at = pc >> 3, cc = pc & 7;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const int key = gw + 4 * m;
          const int sl = 64 * ch + key;
          const int id = (sl < k && sm.idx[sl] >= 0) ? sm.idx[sl] : 0;
          cp_async16_cg(bs + at * 8192 + key * 128 + ((cc ^ (key & 7)) << 4),
                        reinterpret_cast<const uint4*>(kvb + (long long)id * kDQK) + pc);
        }
      }
      cp_async_arrive_noinc(smem_u32(&sm.full[st]));
    }
    cp_async_wait_all();  // no copy may still be in flight when the CTA exits
  } else if (lane == 0) {
    constexpr uint32_t idesc256 = idesc_bf16(128, 256, false, true);
    constexpr uint32_t idesc64 = idesc_bf16(128, 64, false, true);
    for (int ch = 0; ch < nch; ++ch) {
      const int st = ch % kQStages;
      if (!mbar_wait(smem_u32(&sm.full[st]), (ch / kQStages) & 1, c, abort_flag)) break;
      fence_proxy_async_smem();  // the gathered kv rows (cp.async writes) -> tensor cores
      tc_fence_after();
      const uint32_t b0 = smem_u32(sm.bm[st]);
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        const uint32_t a0 = smem_u32(sm.a[st][hl]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc(a0 + kk * 32, 16, 1024, kSw128);
          const uint32_t acc = (ch > 0 || hl > 0 || kk > 0) ? 1u : 0u;
          mma_bf16_ss(tmem, ad, sdesc(b0 + kk * 2048, 8192, 1024, kSw128), idesc256, acc);
          if (natoms == kQAtoms)  // the fifth atom: columns 256..319 of the tile
            mma_bf16_ss(tmem + 256, ad, sdesc(b0 + 4 * 8192 + kk * 2048, 8192, 1024, kSw128), idesc64,
                        acc);
        }
      }
      mma_commit(smem_u32(&sm.empty[st]));
    }
    mma_commit(smem_u32(&sm.done));
  }
  if (warp >= 2) {
    const int quad = warp & 3;
    const int h = quad * 32 + lane;
    bool have = nch > 0 && mbar_wait_warp(smem_u32(&sm.done), 0, c, abort_flag);
    tc_fence_after();
    __nv_bfloat16* dst = dq + (row * kH + h) * (long long)kDQK + col0;
#pragma unroll 1
    for (int cc = 0; cc < natoms * 64; cc += 32) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + cc, v);
        tmem_ld_wait(v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      uint4 pk[4];
      uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
      for (int i = 0; i < 16; ++i) pw[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = pk[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------- dkv --------------------------------------
// Persistent: one CTA per SM walks work items (row, column tile nt: [0,256) |
// [256,512) | [512,576)), item = 3 * row + nt, strided over the grid, so the
// three column tiles of a row run on neighbouring CTAs at about the same time
// and read the row's P / dS tiles once from HBM and twice from L2.
//
// Per item, D[128 keys x N] = (scale*dS)^T Q (+ P^T dO for value columns) for
// every 128-key tile of the row, contracted over the 128 heads in eight
// chunks of 16.  The B operands (q and dO columns of the item, 128 heads x N)
// stay resident in shared memory for all key tiles; the A operands (dS^T and
// P^T as bf16 pairs hi + lo, 128 keys x 16 heads; a single bf16 rounding of P
// or dS would leave the accumulated dKV of early keys about 0.1 off) stream
// through a 4-stage TMA ring.  Both operands are MN-major straight from TMA
// boxes (64 keys or 64 columns by 16 heads).  Two TMEM accumulators of 256
// columns let the four epilogue warps scatter key tile j (fp32 vector
// reductions into dkv, full 128-byte line segments) while the MMAs of key
// tile j + 1 run.  The next item's B chunks reload one by one as the MMAs of
// the current item's last key tile release them.
//
// warp 0 lane 0: MMA issue; warp 1 lane 0: TMA; warps 2-9: TMEM drain and
// scatter (warp w reads TMEM lanes 32 * (w % 4) ..., half (w - 2) / 4 of the
// item's columns: eight warps keep enough reductions in flight).  Key tiles with no
// valid id skip their loads and MMAs (the producer and the issuer derive the
// same tile mask from the index row); the accumulator protocol still runs
// for them and the epilogue adds nothing.
constexpr int kVStages = 4;
constexpr int kVHeads = 16;                 // heads per chunk
constexpr int kVChunks = kH / kVHeads;      // 8
constexpr int kVBox = 64 * kVHeads * 2;     // 2 KB: 64 keys (or columns) x 16 heads
constexpr int kVThreads = 320;
constexpr int kVEpiWarps = 8;
struct __align__(1024) DkvSmem {
  uint8_t bq[kVChunks][4][kVBox];           // q columns of the item, [head chunk][64-column box]
  uint8_t bo[kVChunks][4][kVBox];           // dO columns
  uint8_t a[kVStages][4][2][kVBox];         // [dS hi, dS lo, P hi, P lo][key half]
  uint8_t scratch[kVEpiWarps][4096];        // scatter transpose, one per epilogue warp
  uint64_t afull[kVStages], aempty[kVStages], bfull[kVChunks], bempty[kVChunks];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DkvSmem) + 1024 <= 232448, "dkv shared memory");

// bit j: key tile j of the row holds at least one valid key id (warp-wide)
__device__ __forceinline__ uint32_t dkv_tile_mask(const int32_t* __restrict__ idx_row, int k, int S_k) {
  const int lane = threadIdx.x & 31;
  uint32_t m = 0;
#pragma unroll 16
  for (int sl = lane; sl < k; sl += 32) {
    const int id = idx_row[sl];
    if (id >= 0 && id < S_k) m |= 1u << (sl >> 7);
  }
  return __reduce_or_sync(0xffffffffu, m);
}

__global__ void __launch_bounds__(kVThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_dslo,
               const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_plo,
               const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
               Shape s, const int32_t* __restrict__ idx, float* __restrict__ dkv, int ntile,
               long long nitems, DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  DkvSmem& sm = *reinterpret_cast<DkvSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = s.topk;
  volatile int* abort_flag = &sm.abort;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(smem_u32(&sm.afull[i]), 1);
      mbar_init(smem_u32(&sm.aempty[i]), 1);
    }
    for (int i = 0; i < kVChunks; ++i) {
      mbar_init(smem_u32(&sm.bfull[i]), 1);
      mbar_init(smem_u32(&sm.bempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.acc_full[i]), 1);
      mbar_init(smem_u32(&sm.acc_empty[i]), kVEpiWarps);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;
  if (warp == 0) {
    // ---- MMA issue ----
    uint32_t ast = 0, g = 0, it = 0;
    for (long long item = blockIdx.x; ok && item < nitems; item += gridDim.x, ++it) {
      const long long row = item / 3;
      const int nt = (int)(item % 3);
      const uint32_t mask = dkv_tile_mask(idx + row * k, k, s.S_k);
      if (lane == 0) {
        const int N = nt < 2 ? 256 : 64;
        const int nA = nt < 2 ? 4 : 2;
        const uint32_t idesc = idesc_bf16(128, N, true, true);
        // B chunk ch is awaited at the first valid tile j0, in the order the
        // producer issues it (B chunk ch, then tile j0's A chunk ch), and
        // released after its last reader (chunk ch of the last valid tile
        // jl).  Commits only follow MMAs: a tile without MMAs arrives on its
        // accumulator barrier directly.
        const int j0 = mask ? __ffs(mask) - 1 : -1;
        const int jl = mask ? 31 - __clz(mask) : -1;
        for (int ch = 0; ok && jl < 0 && ch < kVChunks; ++ch) {  // no valid tile: B unused
          ok = mbar_wait(smem_u32(&sm.bfull[ch]), it & 1, c, abort_flag);
          if (ok) mbar_arrive(smem_u32(&sm.bempty[ch]));
        }
        for (int j = 0; ok && j < ntile; ++j, ++g) {
          const uint32_t buf = g & 1;
          ok = mbar_wait(smem_u32(&sm.acc_empty[buf]), ((g >> 1) & 1) ^ 1, c, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const bool valid = (mask >> j) & 1u;
          const uint32_t d = tmem + buf * 256;
          bool first = true;
          for (int ch = 0; valid && ch < kVChunks; ++ch) {
            if (j == j0) {
              ok = mbar_wait(smem_u32(&sm.bfull[ch]), it & 1, c, abort_flag);
              if (!ok) break;
            }
            const uint32_t st = ast % kVStages;
            ok = mbar_wait(smem_u32(&sm.afull[st]), (ast / kVStages) & 1, c, abort_flag);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int o = 0; o < nA; ++o) {
              const uint32_t a0 = smem_u32(sm.a[st][o][0]);
              const uint32_t b0 = smem_u32(o < 2 ? sm.bq[ch][0] : sm.bo[ch][0]);
              mma_bf16_ss(d, sdesc(a0, kVBox, 1024, kSw128), sdesc(b0, kVBox, 1024, kSw128), idesc,
                          first ? 0u : 1u);
              first = false;
            }
            mma_commit(smem_u32(&sm.aempty[st]));
            ++ast;
            if (j == jl) mma_commit(smem_u32(&sm.bempty[ch]));
          }
          if (!ok) break;
          if (valid) mma_commit(smem_u32(&sm.acc_full[buf]));
          else mbar_arrive(smem_u32(&sm.acc_full[buf]));  // nothing to read: the epilogue skips it
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
  } else if (warp == 1) {
    // ---- TMA: B chunks once per item, A chunks per valid key tile ----
    const CUtensorMap* am[4] = {&tm_ds, &tm_dslo, &tm_p, &tm_plo};
    uint32_t ast = 0, it = 0;
    for (long long item = blockIdx.x; ok && item < nitems; item += gridDim.x, ++it) {
      const long long row = item / 3;
      const int nt = (int)(item % 3);
      const uint32_t mask = dkv_tile_mask(idx + row * k, k, s.S_k);
      if (lane == 0) {
        const bool withV = nt < 2;
        const int ncb = withV ? 4 : 1;
        const int nA = withV ? 4 : 2;
        const uint32_t bytesA = (uint32_t)(nA * 2) * kVBox;
        const uint32_t bytesB = (uint32_t)((withV ? 2 : 1) * ncb) * kVBox;
        const int y0 = (int)(row * kH);
        auto load_a = [&](int j, int ch) -> bool {
          const uint32_t st = ast % kVStages;
          if (!mbar_wait(smem_u32(&sm.aempty[st]), ((ast / kVStages) & 1) ^ 1, c, abort_flag)) return false;
          const uint32_t fb = smem_u32(&sm.afull[st]);
          mbar_arrive_expect_tx(fb, bytesA);
          for (int o = 0; o < nA; ++o)
            for (int kk = 0; kk < 2; ++kk)
              tma_load_2d(smem_u32(sm.a[st][o][kk]), am[o], j * 128 + 64 * kk, y0 + kVHeads * ch, fb);
          ++ast;
          return true;
        };
        const int j0 = mask ? __ffs(mask) - 1 : -1;
        for (int ch = 0; ok && ch < kVChunks; ++ch) {
          ok = mbar_wait(smem_u32(&sm.bempty[ch]), (it & 1) ^ 1, c, abort_flag);
          if (!ok) break;
          const uint32_t fb = smem_u32(&sm.bfull[ch]);
          mbar_arrive_expect_tx(fb, bytesB);
          for (int cb = 0; cb < ncb; ++cb) {
            tma_load_2d(smem_u32(sm.bq[ch][cb]), &tm_q, 256 * nt + 64 * cb, y0 + kVHeads * ch, fb);
            if (withV) tma_load_2d(smem_u32(sm.bo[ch][cb]), &tm_do, 256 * nt + 64 * cb, y0 + kVHeads * ch, fb);
          }
          if (j0 >= 0) ok = load_a(j0, ch);
        }
        for (int j = j0 + 1; ok && j0 >= 0 && j < ntile; ++j)
          if ((mask >> j) & 1u)
            for (int ch = 0; ok && ch < kVChunks; ++ch) ok = load_a(j, ch);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
  } else {
    // ---- TMEM drain and scatter: thread = key of the tile ----
    const int quad = warp & 3, half = (warp - 2) >> 2;
    const uint32_t scratch = smem_u32(sm.scratch[warp - 2]);
    uint32_t g = 0;
    for (long long item = blockIdx.x; ok && item < nitems; item += gridDim.x) {
      const long long row = item / 3;
      const int nt = (int)(item % 3);
      const int N = nt < 2 ? 256 : 64;
      const long long b = row / s.S_q;
      for (int j = 0; ok && j < ntile; ++j, ++g) {
        const uint32_t buf = g & 1;
        const int sl = j * 128 + quad * 32 + lane;
        int id = sl < k ? idx[row * k + sl] : -1;
        if (id >= s.S_k) id = -1;
        ok = mbar_wait_warp(smem_u32(&sm.acc_full[buf]), (g >> 1) & 1, c, abort_flag);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, id >= 0)) {
          float* dst = id < 0 ? nullptr : dkv + (b * s.S_k + id) * (long long)kDQK + 256 * nt;
          const uint32_t taddr = tmem + buf * 256 + ((uint32_t)(quad * 32) << 16);
          const int c1 = (half + 1) * (N / 2);
#pragma unroll 1
          for (int cc = half * (N / 2); cc < c1; cc += 64) {
            const bool two = cc + 32 < c1;
            uint32_t v[32], w[32];
            tmem_ld32(taddr + cc, v);
            if (two) tmem_ld32(taddr + cc + 32, w);
            tmem_ld_wait(v);
            warp_scatter_add_32x32(scratch, v, dst == nullptr ? nullptr : dst + cc);
            if (two) {
              tmem_ld_also(w);
              warp_scatter_add_32x32(scratch, w, dst == nullptr ? nullptr : dst + cc + 32);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[buf]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace bwd

bool make_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

// workspace layout of the bf16 attention backward: P_hi, P_lo,
// (scale*dS)_hi, (scale*dS)_lo [rows*128][k] bf16, then D [rows*128] fp32
size_t bwd_tc_workspace(const Shape& s) {
  const size_t rh = (size_t)s.B * s.S_q * bwd::kH;
  return 4 * rh * (size_t)s.topk * 2 + rh * 4 + 256;
}
// the KL pass: head-summed attention probabilities [rows][k] fp32
size_t kl_tc_workspace(const Shape& s) {
  const size_t rows = (size_t)s.B * s.S_q;
  return rows * (size_t)s.topk * 4 + 256;
}

int launch_kl_tc(const Shape& s, const void* q_I, const void* k_I, const void* w,
                 const int32_t* idx, const float* praw, float* loss, void* dq_I, float* dk_I,
                 float* dw, DevCtx c, cudaStream_t st);

template <typename K>
static bool set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
         cudaSuccess;
}

// praw (optional, [rows][k] fp32): also write the head-summed probabilities
// the indexer KL loss takes as its target
int launch_attn_bwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx,
                       const void* out, const void* dout, const float* mx, const float* sm,
                       void* dq, float* dkv, void* ws, DevCtx c, cudaStream_t st,
                       float* praw) {
  using namespace bwd;
  const long long rows = (long long)s.B * s.S_q, rh = rows * kH;
  const int k = s.topk;
  __nv_bfloat16* P_ws = (__nv_bfloat16*)ws;
  __nv_bfloat16* Plo_ws = P_ws + rh * k;
  __nv_bfloat16* dS_ws = Plo_ws + rh * k;
  __nv_bfloat16* dSlo_ws = dS_ws + rh * k;
  float* D = (float*)(dSlo_ws + rh * k);
  const int ntile = (k + 127) / 128;
  // D = rowsum(dO * O)
  rowdot_kernel<<<(unsigned)((rh * 32 + 255) / 256), 256, 0, st>>>(
      (const __nv_bfloat16*)dout, (const __nv_bfloat16*)out, D, rh);
  CUtensorMap tq, tdo, tds, tdslo, tds2, tdslo2, tp2, tplo2, tq2, tdo2;
  if (!make_tmap_2d_bf16(&tq, q, rh, kDQK, 64, kH, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tdo, dout, rh, kDV, 64, kH, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tds, dS_ws, rh, k, 64, kH, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tdslo, dSlo_ws, rh, k, 64, kH, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tds2, dS_ws, rh, k, 64, kVHeads, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tdslo2, dSlo_ws, rh, k, 64, kVHeads, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tp2, P_ws, rh, k, 64, kVHeads, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tplo2, Plo_ws, rh, k, 64, kVHeads, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tq2, q, rh, kDQK, 64, kVHeads, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tdo2, dout, rh, kDV, 64, kVHeads, 128)) return DSA_ERR_CUDA;
  const size_t s1 = sizeof(ScoresSmem) + 1024, s2 = sizeof(DqSmem) + 1024, s3 = sizeof(DkvSmem) + 1024;
  if (!set_smem(scores_kernel<true>, s1) || !set_smem(dq_kernel, s2) || !set_smem(dkv_kernel, s3))
    return DSA_ERR_CUDA;
  scores_kernel<true><<<(unsigned)(rows * ntile), kSThreads, s1, st>>>(
      tq, tdo, (const __nv_bfloat16*)kv, s, idx, mx, sm, D, P_ws, Plo_ws, dS_ws, dSlo_ws, praw,
      ntile, c);
  dq_kernel<<<(unsigned)(rows * 2), 192, s2, st>>>(tds, tdslo, (const __nv_bfloat16*)kv, s, idx,
                                                    (__nv_bfloat16*)dq, c);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return DSA_ERR_CUDA;
  const long long nitems = rows * 3;
  dkv_kernel<<<(unsigned)(nitems < sms ? nitems : sms), kVThreads, s3, st>>>(
      tds2, tdslo2, tp2, tplo2, tq2, tdo2, s, idx, dkv, ntile, nitems, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_kl_bwd_tc(const Shape& s, const void* q, const void* kv, const void* q_I,
                     const void* k_I, const void* w, const int32_t* idx, const float* mx,
                     const float* sm, float* loss, void* dq_I, float* dk_I, float* dw, void* ws,
                     DevCtx c, cudaStream_t st) {
  using namespace bwd;
  const long long rows = (long long)s.B * s.S_q, rh = rows * kH;
  const int k = s.topk;
  float* praw = (float*)ws;
  const int ntile = (k + 127) / 128;
  CUtensorMap tq;
  if (!make_tmap_2d_bf16(&tq, q, rh, kDQK, 64, kH, 128)) return DSA_ERR_CUDA;
  const size_t s1 = sizeof(ScoresSmem) + 1024;
  if (!set_smem(scores_kernel<false>, s1)) return DSA_ERR_CUDA;
  scores_kernel<false><<<(unsigned)(rows * ntile), kSThreads, s1, st>>>(
      tq, tq, (const __nv_bfloat16*)kv, s, idx, mx, sm, nullptr, nullptr, nullptr, nullptr, nullptr,
      praw, ntile, c);
  if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  return launch_kl_tc(s, q_I, k_I, w, idx, praw, loss, dq_I, dk_I, dw, c, st);
}

// Attention backward and indexer KL backward sharing one recompute of P: the
// attention pass writes the head-summed probabilities, the KL pass reads them.
int launch_dsa_bwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx,
                      const void* out, const void* dout, const float* mx, const float* sm,
                      const void* q_I, const void* k_I, const void* w, void* dq, float* dkv,
                      float* loss, void* dq_I, float* dk_I, float* dw, void* ws, DevCtx c,
                      cudaStream_t st) {
  float* praw = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + bwd_tc_workspace(s));
  const int rc = launch_attn_bwd_tc(s, q, kv, idx, out, dout, mx, sm, dq, dkv, ws, c, st, praw);
  if (rc) return rc;
  return launch_kl_tc(s, q_I, k_I, w, idx, praw, loss, dq_I, dk_I, dw, c, st);
}

}  // namespace dsa
