// Lightning Indexer scores on FP8 (E4M3) operands, tcgen05 kind::f8f6f4 (sm_103a).
//
// [DSA-32K] Lightning Indexer forward: I[t,s] = sum_j w[t,j] ReLU(q_I[t,j].k_I[s]).
// The pages give no DSA FP8 recipe; this path takes one reading: q_I and k_I
// are quantized per 128-element vector to E4M3 (scale = absmax / 448 in fp32,
// x / scale rounded to nearest even, clamped to +-448: quant_e4m3_kernel) and
// the score is the formula on the dequantized vectors,
//   I[t,s] = sk[s] * sum_j (w[t,j] * sq[t,j]) * ReLU(q8[t,j] . k8[s])
// (the scales are positive, so they move outside the ReLU).  The E4M3
// products are exact and the dot products accumulate in fp32 in TMEM.
//
// Same tiling as the bf16 kernel (indexer_tc.cu): one MMA computes
// D[128 keys x 256] = k8[128 keys x 128] * q8[4 tokens x 64 heads x 128]^T
// (M = 128, N = 256, K = 32 per instruction, 4 instructions per key block),
// TMEM lane = key; a CTA owns 4 query rows (B operand resident, 32 KB) and
// streams 128-key blocks of k8 (16 KB) through a TMA ring; two 256-column
// accumulators overlap the epilogue of block i with the MMA of block i+1.
//
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..9 = epilogue (two warps per TMEM lane quadrant, two tokens each).
#include <math.h>

#include <cuda_fp8.h>

#include "dsa_common.cuh"

namespace dsa {
namespace idxf8 {

constexpr int kHI = 64, kDI = 128;
constexpr int kTQ = 4;                    // query rows per CTA tile
constexpr int kN = kTQ * kHI;             // 256: MMA N
constexpr int kBK = 128;                  // keys per block: MMA M
constexpr int kStages = 6;
constexpr int kAStage = kBK * 128;        // 128 keys x 128 dims, E4M3, SW128: 16 KB
constexpr int kBBytes = kN * 128;         // 256 rows x 128 dims: 32 KB
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kTmemCols = 512;
// kind::f8f6f4 instruction descriptor: D fp32, A and B E4M3 (format 0), both
// K-major, N >> 3, M >> 4
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kBK >> 4) << 24);

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct __align__(1024) Smem {
  uint8_t a[kStages][kAStage];
  uint8_t b[kBBytes];
  float w[kTQ][kHI];
  long long pos[kTQ];
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], b_full, mma_done;
  uint32_t tmem_base;
  int abort;
  int nkb;
};

__global__ void __launch_bounds__(kThreads, 1)
    indexer_f8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      Shape s, const __nv_bfloat16* __restrict__ w, const float* __restrict__ q_scale,
                      const float* __restrict__ k_scale, long long row_lo, long long row_hi,
                      long long row_begin, int batch, float* __restrict__ scores, long long ld,
                      DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long ntiles = (row_hi - row_lo + kTQ - 1) / kTQ;
  const long long tile = ntiles - 1 - blockIdx.x;  // heaviest (latest) rows first
  const long long r0 = row_lo + tile * kTQ;        // first flattened row of the tile
  volatile int* abort_flag = &sm.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1);
      mbar_init(smem_u32(&sm.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.acc_full[i]), 1);
      mbar_init(smem_u32(&sm.acc_empty[i]), kEpiWarps * 32);
    }
    mbar_init(smem_u32(&sm.b_full), 1);
    mbar_init(smem_u32(&sm.mma_done), 1);
    sm.abort = 0;
    long long maxpos = -1;
    for (int j = 0; j < kTQ; ++j) {
      const long long row = r0 + j;
      long long p = -1;
      if (row < row_hi) {
        p = row_pos(s, row);
        if (p < 0 || p >= s.S_k) {
          set_status(c, DSA_ERR_INDEX);
          p = -1;
        }
      }
      sm.pos[j] = p;
      maxpos = p > maxpos ? p : maxpos;
    }
    sm.nkb = (int)((maxpos + kBK) / kBK);  // 0 when no row is valid
    fence_mbar_init();
  }
  if (threadIdx.x >= 64) {
    const int e = threadIdx.x - 64;  // 256 epilogue threads load w for the 4 rows
    const int j = e / kHI, h = e % kHI;
    const long long row = r0 + j;
    // the query scale moves into the head weight: w[t,j] * sq[t,j]
    sm.w[j][h] = row < row_hi ? __bfloat162float(w[row * kHI + h]) * q_scale[row * kHI + h] : 0.f;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int nkb = sm.nkb;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && nkb > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      const uint32_t bf = smem_u32(&sm.b_full);
      mbar_arrive_expect_tx(bf, kBBytes);
      const int qrow = (int)(r0 * kHI);
      tma_load_2d(smem_u32(sm.b), &tm_q, 0, qrow, bf);
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int st = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        if (!mbar_wait(smem_u32(&sm.empty[st]), ph ^ 1, c, abort_flag)) break;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, kAStage);
        const int krow = (int)((long long)batch * s.S_k + (long long)kb * kBK);
        tma_load_2d(smem_u32(sm.a[st]), &tm_k, 0, krow, fb);
      }
      // drain: every issued load has landed before the CTA may exit
      mbar_wait(bf, 0, c, abort_flag);
      for (int i = (kb > kStages ? kb - kStages : 0); i < kb; ++i)
        mbar_wait(smem_u32(&sm.full[i % kStages]), (i / kStages) & 1, c, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0 && nkb > 0) {
      bool ok = mbar_wait(smem_u32(&sm.b_full), 0, c, abort_flag);
      tc_fence_after();
      const uint32_t b0 = smem_u32(sm.b);
      for (int kb = 0; ok && kb < nkb; ++kb) {
        const int st = kb % kStages, acc = kb & 1;
        if (!mbar_wait(smem_u32(&sm.acc_empty[acc]), ((kb >> 1) & 1) ^ 1, c, abort_flag)) break;
        if (!mbar_wait(smem_u32(&sm.full[st]), (kb / kStages) & 1, c, abort_flag)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(sm.a[st]);
        const uint32_t d = tmem + acc * kN;
#pragma unroll
        for (int k = 0; k < kDI / 32; ++k) {  // 32 E4M3 elements = 32 bytes per step
          const uint64_t ad = sdesc(a0 + k * 32, 16, 1024, kSw128);
          const uint64_t bd = sdesc(b0 + k * 32, 16, 1024, kSw128);
          mma_f8_ss(d, ad, bd, kIdesc, k > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.empty[st]));
        mma_commit(smem_u32(&sm.acc_full[acc]));
      }
      mma_commit(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0, c, abort_flag);
    }
  } else {
    // -------------------------------- epilogue --------------------------------
    const int ew = warp - 2;
    const int quad = warp & 3;       // TMEM lanes this warp may access
    const int half = ew >> 2;        // tokens {2*half, 2*half+1}
    for (int kb = 0; kb < nkb; ++kb) {
      const int acc = kb & 1;
      if (!mbar_wait_warp(smem_u32(&sm.acc_full[acc]), (kb >> 1) & 1, c, abort_flag)) break;
      tc_fence_after();
      const long long key = (long long)kb * kBK + quad * 32 + lane;
      const float skey = key < s.S_k ? k_scale[(long long)batch * s.S_k + key] : 0.f;
      // both tokens of the warp (2*half, 2*half+1): pipelined TMEM loads
      const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + acc * kN + half * 2 * kHI;
      uint32_t A[32], B[32];
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int j = half * 2 + tt;
        const float sc = tt == 0 ? relu_pair_first(tb, sm.w[j], A, B) : relu_pair_second(tb, sm.w[j], A, B);
        if (key <= sm.pos[j]) scores[(r0 + j - row_begin) * ld + key] = skey * sc;
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.acc_empty[acc]));
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// quantize rows of 128 bf16 values to E4M3 with one fp32 scale per row:
// one warp per row, 4 values per lane
__global__ void quant_e4m3_kernel(const __nv_bfloat16* __restrict__ x, long long nrows,
                                  uint8_t* __restrict__ q, float* __restrict__ scale) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + row * 128 + 4 * lane);
  const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  const float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax > 0.f ? amax / 448.f : 1.f;  // IEEE division
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8_storage_t code = __nv_cvt_float_to_fp8(v[i] / sc, __NV_SATFINITE, __NV_E4M3);
    packed |= (uint32_t)code << (8 * i);
  }
  reinterpret_cast<uint32_t*>(q + row * 128)[lane] = packed;
  if (lane == 0) scale[row] = sc;
}

}  // namespace idxf8

bool make_tmap_2d_u8(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                     uint32_t box_rows);

int launch_quant_e4m3(const void* x, long long nrows, uint8_t* q, float* scale, cudaStream_t st) {
  if (nrows <= 0) return DSA_OK;
  const int warps = 8;
  idxf8::quant_e4m3_kernel<<<(unsigned)((nrows + warps - 1) / warps), warps * 32, 0, st>>>(
      (const __nv_bfloat16*)x, nrows, q, scale);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_indexer_f8(const Shape& s, const uint8_t* q8, const float* q_scale, const uint8_t* k8,
                      const float* k_scale, const void* w, long long row_begin, long long rows,
                      float* scores, long long ld, DevCtx c, cudaStream_t st) {
  using namespace idxf8;
  CUtensorMap tq, tk;
  if (!make_tmap_2d_u8(&tq, q8, (uint64_t)s.B * s.S_q * kHI, kDI, kDI, kN)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_u8(&tk, k8, (uint64_t)s.B * s.S_k, kDI, kDI, kBK)) return DSA_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  if (cudaFuncSetAttribute(indexer_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long r_end = row_begin + rows;
  for (int b = 0; b < s.B; ++b) {
    const long long lo = row_begin > (long long)b * s.S_q ? row_begin : (long long)b * s.S_q;
    const long long hi = r_end < (long long)(b + 1) * s.S_q ? r_end : (long long)(b + 1) * s.S_q;
    if (hi <= lo) continue;
    const long long ntiles = (hi - lo + kTQ - 1) / kTQ;
    indexer_f8_kernel<<<(unsigned)ntiles, kThreads, smem, st>>>(
        tq, tk, s, (const __nv_bfloat16*)w, q_scale, k_scale, lo, hi, row_begin, b, scores, ld, c);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // namespace dsa
