// Sparse multi-query attention forward on tcgen05 (bf16 in, fp32 accumulate).
//
// [DSA-32K] Sparse Flash Attention forward: p[t] = Softmax(q[t] K_topk^T scale),
// O[t] = p[t] V_topk; the 128 heads of token t share its top-k kv rows, each
// row 576 wide (512 latent + 64 rope) and V = its first 512 columns
// (weight-absorbed MLA).
//
// One token per CTA pair (a cluster of two).  Moving the selected kv rows from
// L2 into shared memory is the bound of this kernel (about 18-24 bytes per
// cycle per SM through cp.async, whatever the access pattern), so each row is
// gathered once per pair: CTA c gathers its 288 columns of every selected row,
// D_c = value columns E_c = [128c, 128c+128) u [256+128c, 256+128c+128) plus
// rope columns [512+32c, 512+32c+32).  Nothing else crosses between the CTAs
// through the cp.async / st.async path.
//
// Every MMA is a two-CTA MMA (cta_group::2, M = 128 = 64 rows per CTA,
// N = 256) issued by CTA 0.  B is split by N between the CTAs' shared
// memories, and each CTA's accumulator keeps its 64 rows twice over the 128
// TMEM lanes: lanes 0..63 pair with CTA 0's half of B, lanes 64..127 with CTA
// 1's half.  With A in TMEM, lanes 0..63 and 64..127 of A may hold different
// data, which splits the logit contraction between the CTAs without any
// exchange.  CTA c owns heads [64c, 64c+64).  Per 128-slot block:
//   1. logits, 16 steps with A in TMEM: lanes h / 64+h of A hold head h's
//      query columns E_0 / E_1; B rows n < 128 are CTA 0's columns E_0 of slot
//      n, rows n >= 128 CTA 1's columns E_1 of slot n - 128.  Then 4 rope
//      steps with A = the head's 64 rope columns in shared memory and B the
//      rope area, whose columns 32c..32c+31 hold CTA c's rope data and the
//      other 32 zeros.  Lane h of the accumulator ends with head h's partial
//      logit over D_0 for the 128 slots, lane 64+h with the partial over D_1;
//   2. the two halves are added through shared memory (each thread of a lane
//      pair keeps 32 slots), then the fp32 online softmax (exp2 domain; the
//      running max used for P only moves when a head's block max exceeds it
//      by more than 2^8, so the O rescale in TMEM is rare) and P as bf16 into
//      shared memory (K-major: row = head, slots contiguous);
//   3. O += P V with N = 256 value columns: B rows n < 128 = CTA 0's value
//      columns, n >= 128 CTA 1's, both from the gathered block (no second
//      gather of V); two MMAs per 16-slot step cover the 512 columns.  O of
//      the CTA's 64 heads takes 256 TMEM columns: O column 128m + i of lane h
//      is value column 256m + i, of lane 64 + h value column 256m + 128 + i.
// Two block stages in shared memory (cp.async gathers completing on the
// stage barrier); the MMA order is S(0), PV(0), S(1), PV(1), ...
//
// Roles per CTA: warp 0 = TMEM allocation, the MMA issuer in CTA 0 and the
// readiness relay in CTA 1 (CTA 0 must know when CTA 1's operands are ready:
// the relay waits on CTA 1's local barriers and arrives on CTA 0's); warps
// 1..4 = kv gather (warp 1 also TMA-loads the rope query columns); warps
// 5..12 = query columns into TMEM, then softmax and epilogue (warp w: TMEM
// lane quadrant w % 4, logit columns [64ch, 64ch+64) with ch = (w - 5) / 4).
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace attn {

constexpr int kH = 128, kHC = 64, kDQK = 576, kDV = 512;
constexpr int kBlk = 128;                          // slots per block
constexpr int kMaxTopk = 2048;
constexpr int kStages = 2;                         // gathered blocks in shared memory
constexpr int kChunk = kBlk * 128;                 // 128 slots x 64 columns (SW128 rows)
constexpr int kStageBytes = 5 * kChunk;            // 4 value chunks + the rope area
constexpr int kGatherWarps = 4, kSoftWarps = 8;
constexpr int kWarpGather0 = 1, kWarpSoft0 = kWarpGather0 + kGatherWarps;
constexpr int kThreads = 32 * (1 + kGatherWarps + kSoftWarps);
constexpr int kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;
constexpr uint32_t kIdescS = idesc_bf16(128, 256, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);
constexpr float kRescaleThreshold = 8.0f;          // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct __align__(1024) Smem {
  uint8_t stage[kStages][kStageBytes];             // [value chunk 0..3 | rope area][slot][128 B]
  uint8_t qrope[kHC * 128];                        // rope query columns, K-major SW128
  uint8_t p[kBlk / 64][kHC * 128];                 // P: 2 chunks of 64 slots, K-major SW128
  float4 xbuf[2][2][8][kHC];                       // partial-logit exchange [ch][dest half][i][head]
  unsigned long long mask[kMaxTopk / 64];          // per 64 slots: valid slots
  float red[kSoftWarps][32];                       // per-warp partial block maxima / row sums
  uint64_t st_full[kStages], st_empty[kStages];
  uint64_t q_full, q_tm, q_peer, s_full, p_full, mma_done;
  uint32_t tmem_base;
  int abort;
  int last;
  int bad;
};
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- two-CTA (cta_group::2) tcgen05 forms: every tcgen05 instruction of this
// kernel that takes a CTA group uses ::2 ----
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma2_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// arrive once on the barrier at the same offset in both CTAs of the pair when
// every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void commit2(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
// arrive on a barrier of the peer CTA, ordering this thread's earlier memory
// operations (and what it observed) before the arrive at cluster scope
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const void* __restrict__ qg,
                       const void* __restrict__ kvg, Shape s, const int32_t* __restrict__ idx,
                       __nv_bfloat16* __restrict__ out, float* __restrict__ mx,
                       float* __restrict__ sm_out, long long nrows, DevCtx c) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const long long row = nrows - 1 - (long long)(blockIdx.x >> 1);  // flattened query row
  const long long b = row / s.S_q;
  const int k = s.topk;
  const int32_t* irow = idx + row * (long long)k;
  volatile int* abort_flag = &sm.abort;

  if (threadIdx.x == 32 * kWarpGather0) {
    // CTA 0's stage barriers also count the relay's arrive for CTA 1's stage
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.st_full[i]), kGatherWarps * 32 + (crank == 0 ? 1 : 0));
      mbar_init(smem_u32(&sm.st_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.q_tm), kSoftWarps);
    mbar_init(smem_u32(&sm.q_peer), 1);
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.p_full), 2 * kSoftWarps);  // (used in CTA 0) both CTAs' softmax warps
    mbar_init(smem_u32(&sm.mma_done), 1);
    sm.abort = 0;
    sm.last = -1;
    sm.bad = 0;
    fence_mbar_init();
    // the rope query columns of this CTA's 64 heads: one 64 x 64 box (SW128)
    tma_prefetch_desc(&tm_q);
    const uint32_t qb = smem_u32(&sm.q_full);
    mbar_arrive_expect_tx(qb, kHC * 128);
    tma_load_2d(smem_u32(sm.qrope), &tm_q, kDV, (int)(row * kH + kHC * crank), qb);
  }
  if (warp == 0) {
    tmem_alloc2(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish2();
    tc_fence_before();
  }
  // the other CTA's half of both rope areas: zeros, for the whole kernel
  for (int i = threadIdx.x; i < kStages * kBlk * 4; i += kThreads) {
    const int st = i / (kBlk * 4), r = (i >> 2) % kBlk, pc = 4 * (1 - (int)crank) + (i & 3);
    *reinterpret_cast<uint4*>(sm.stage[st] + 4 * kChunk + r * 128 + ((pc ^ (r & 7)) << 4)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  // scan the index row: last valid slot, out-of-range entries (skipped, reported)
  int last = -1, bad = 0;
  for (int i = threadIdx.x; i < k; i += kThreads) {
    const int id = irow[i];
    if (id < -1 || id >= s.S_k) bad = 1;
    else if (id >= 0) last = i;
  }
  __syncthreads();  // barrier init (sm.last / sm.bad) visible
  if (last >= 0) atomicMax(&sm.last, last);
  if (bad) sm.bad = 1;
  __syncthreads();
  const int nblk = (sm.last + kBlk) / kBlk;
  for (int g = warp; g < nblk * (kBlk / 64); g += kThreads / 32) {
    const int s0 = g * 64 + lane, s1 = s0 + 32;
    const int i0 = s0 < k ? irow[s0] : -1, i1 = s1 < k ? irow[s1] : -1;
    const uint32_t lo = __ballot_sync(0xffffffffu, i0 >= 0 && i0 < s.S_k);
    const uint32_t hi = __ballot_sync(0xffffffffu, i1 >= 0 && i1 < s.S_k);
    if (lane == 0) sm.mask[g] = ((unsigned long long)hi << 32) | lo;
  }
  if (threadIdx.x == 0 && sm.bad) set_status(c, DSA_ERR_INDEX);
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp >= kWarpGather0 && warp < kWarpSoft0) {
    // ------------------------------- kv gather -------------------------------
    // Warp gw gathers slots [32gw, 32gw+32) of each block.  Value columns: one
    // warp-wide copy per slot, lanes 0..15 the 256 contiguous bytes of columns
    // [128c, 128c+128), lanes 16..31 those of [256+128c, 256+128c+128), into
    // value chunks 0..3 (SW128 rows).  Rope: 8 slots per copy, 4 lanes per
    // slot, into this CTA's half of the rope area.  Invalid slots copy row 0,
    // so every byte the MMAs read is finite (their P is 0).
    const int gw = warp - kWarpGather0;
    const __nv_bfloat16* kvb = reinterpret_cast<const __nv_bfloat16*>(kvg) + b * s.S_k * (long long)kDQK;
    const int run = lane >> 4, p16 = lane & 15;
    const int vcol = 256 * run + 128 * (int)crank + 8 * p16;   // this lane's value piece
    const int vchunk = 2 * run + (p16 >> 3), vpc = p16 & 7;
    const int rs = lane >> 2, rp = lane & 3;                   // rope: slot in group of 8, piece
    const int rcol = kDV + 32 * (int)crank + 8 * rp, rpc = 4 * (int)crank + rp;
    for (int j = 0; j < nblk; ++j) {
      const int st = j % kStages;
      // this warp's 32 indices of the block (loaded before the wait)
      const int e = j * kBlk + 32 * gw + lane;
      int id = e < k ? irow[e] : -1;
      if (id < 0 || id >= s.S_k) id = 0;
      if (!mbar_wait_warp(smem_u32(&sm.st_empty[st]), ((j / kStages) & 1) ^ 1, c, abort_flag)) break;
      const uint32_t base = smem_u32(sm.stage[st]);
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * gw + i;
        const int rid = __shfl_sync(0xffffffffu, id, i);
        cp_async16_cg(base + vchunk * kChunk + r * 128 + ((vpc ^ (r & 7)) << 4),
                      kvb + (long long)rid * kDQK + vcol);
      }
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        const int rl = 8 * g8 + rs;
        const int r = 32 * gw + rl;
        const int rid = __shfl_sync(0xffffffffu, id, rl);
        cp_async16_cg(base + 4 * kChunk + r * 128 + ((rpc ^ (r & 7)) << 4),
                      kvb + (long long)rid * kDQK + rcol);
      }
      cp_async_arrive_noinc(smem_u32(&sm.st_full[st]));
    }
    cp_async_wait_all();  // no copy may still be in flight when the CTA exits
    if (warp == kWarpGather0 && lane == 0) mbar_wait(smem_u32(&sm.q_full), 0, c, abort_flag);
  } else if (warp == 0) {
    if (crank == 0 && lane == 0 && nblk > 0) {
      // ------------------------------- MMA issuer -------------------------------
      bool ok = mbar_wait(smem_u32(&sm.q_full), 0, c, abort_flag) &&
                mbar_wait(smem_u32(&sm.q_tm), 0, c, abort_flag) &&
                mbar_wait<true>(smem_u32(&sm.q_peer), 0, c, abort_flag);
      tc_fence_after();
      const uint32_t qr = smem_u32(sm.qrope), p0 = smem_u32(sm.p[0]);
      for (int j = 0; ok && j < nblk; ++j) {
        const int st = j % kStages;
        if (!mbar_wait<true>(smem_u32(&sm.st_full[st]), (j / kStages) & 1, c, abort_flag)) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();  // the gathered block (cp.async writes) -> tensor cores
        tc_fence_after();
        const uint32_t sb = smem_u32(sm.stage[st]);
        // S(j): 16 value-column steps (A in TMEM, different in the two lane
        // halves), then 4 rope steps (A in shared memory).  The softmax warps
        // have read S(j-1): PV(j-1) waited for their P.
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          mma2_ts(tmem + kColS, tmem + kColQ + kk * 8,
                  sdesc(sb + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024, kSw128), kIdescS,
                  kk > 0 ? 1u : 0u);
#pragma unroll
        for (int r = 0; r < 4; ++r)
          mma2_ss(tmem + kColS, sdesc(qr + r * 32, 16, 1024, kSw128),
                  sdesc(sb + 4 * kChunk + r * 32, 16, 1024, kSw128), kIdescS, 1u);
        commit2(smem_u32(&sm.s_full));
        // PV(j): both CTAs' P written (and O rescaled if needed)
        if (!mbar_wait<true>(smem_u32(&sm.p_full), j & 1, c, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk) {
          const uint64_t ad = sdesc(p0 + (kk >> 2) * (kHC * 128) + (kk & 3) * 32, 16, 1024, kSw128);
#pragma unroll
          for (int m = 0; m < 2; ++m)
            mma2_ss(tmem + kColO + 128 * m, ad,
                    sdesc(sb + 2 * m * kChunk + kk * 2048, kChunk, 1024, kSw128), kIdescPV,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        commit2(smem_u32(&sm.st_empty[st]));
      }
      commit2(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0, c, abort_flag);
    } else if (crank == 1 && lane == 0 && nblk > 0) {
      // --------------------- readiness relay (CTA 1 -> CTA 0) ---------------------
      if (mbar_wait(smem_u32(&sm.q_full), 0, c, abort_flag) &&
          mbar_wait(smem_u32(&sm.q_tm), 0, c, abort_flag)) {
        tc_fence_after();
        fence_proxy_async_smem();
        mbar_arrive_remote(mapa_shared(smem_u32(&sm.q_peer), 0));
        for (int j = 0; j < nblk; ++j) {
          const int st = j % kStages;
          if (!mbar_wait(smem_u32(&sm.st_full[st]), (j / kStages) & 1, c, abort_flag)) break;
          fence_proxy_async_smem();
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.st_full[st]), 0));
        }
      }
    }
  } else {
    // --------------------------- softmax / epilogue ---------------------------
    // a warp reaches only the TMEM lane quadrant (warp id % 4)
    const int quad = warp & 3, ch = (warp - kWarpSoft0) >> 2;
    const int ws = 4 * ch + quad;                       // slot in red[]
    const int l = quad * 32 + lane;                     // TMEM lane
    const int hl = l & 63, half = l >> 6;               // head in the CTA; lane half
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float sl2e = s.scale * kLog2e;
    float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
    const uint32_t pfull_b = crank == 0 ? smem_u32(&sm.p_full) : mapa_shared(smem_u32(&sm.p_full), 0);
    {
      // query columns of head hl for lane half `half`: E_half's run ch (128
      // columns, contiguous) into TMEM columns kColQ + 64ch .. +64
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(qg) + (row * kH + kHC * crank + hl) * (long long)kDQK +
          256 * ch + 128 * half);
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v4 = __ldg(src + 8 * cc + i);
          w[4 * i] = v4.x;
          w[4 * i + 1] = v4.y;
          w[4 * i + 2] = v4.z;
          w[4 * i + 3] = v4.w;
        }
        tmem_st32(tmem + lane_off + kColQ + 64 * ch + 32 * cc, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.q_tm));
    }
    // The 8 softmax warps synchronise with each other through named barrier
    // 1 (bar.sync, 256 threads): every warp executes the same sequence of
    // barriers whatever happens (after a failed wait it keeps going through
    // the loop without work), so they cannot deadlock.
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      if (ok) ok = mbar_wait_warp(smem_u32(&sm.s_full), j & 1, c, abort_flag);
      // partial logits of head hl over this lane half's columns, slots
      // [64ch, 64ch+64) of the block
      uint32_t v[2][32];
      if (ok) {
        tc_fence_after();
        const uint32_t sbuf = tmem + lane_off + kColS + 64 * ch;
        tmem_ld32(sbuf, v[0]);
        tmem_ld32(sbuf + 32, v[1]);
        tmem_ld_wait(v[0]);
        tmem_ld_also(v[1]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[0][i] = v[1][i] = 0u;
      }
      // keep slots [64ch + 32half, +32): send the other 32 partials to the
      // lane-pair partner (lane l ^ 64, same column half) and add its partials
      // (half is the same in the whole warp; selects keep v in registers)
      uint32_t mine[32], give[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        mine[i] = half ? v[1][i] : v[0][i];
        give[i] = half ? v[0][i] : v[1][i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        sm.xbuf[ch][half ^ 1][i][hl] = make_float4(__uint_as_float(give[4 * i]), __uint_as_float(give[4 * i + 1]),
                                                   __uint_as_float(give[4 * i + 2]), __uint_as_float(give[4 * i + 3]));
      named_bar_sync(1, kSoftWarps * 32);
      float x[32];
      const unsigned long long vmask = sm.mask[2 * j + ch] >> (32 * half);
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 pr = sm.xbuf[ch][half][i][hl];
        x[4 * i] = __uint_as_float(mine[4 * i]) + pr.x;
        x[4 * i + 1] = __uint_as_float(mine[4 * i + 1]) + pr.y;
        x[4 * i + 2] = __uint_as_float(mine[4 * i + 2]) + pr.z;
        x[4 * i + 3] = __uint_as_float(mine[4 * i + 3]) + pr.w;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (((vmask >> i) & 1ull) == 0) x[i] = -INFINITY;
        bm = fmaxf(bm, x[i]);
      }
      // the head's block max over its four threads (lane pair x column halves)
      sm.red[ws][lane] = bm;
      named_bar_sync(1, kSoftWarps * 32);
      bm = fmaxf(fmaxf(sm.red[quad][lane], sm.red[quad + 4][lane]),
                 fmaxf(sm.red[quad ^ 2][lane], sm.red[(quad ^ 2) + 4][lane]));
      // (the next writes of xbuf / red come after the next block's first
      // barrier, which every warp reaches only after these reads)
      if (!ok) continue;
      bm *= sl2e;                                        // log2 units (sl2e > 0)
      m_true = fmaxf(m_true, bm);
      // the same decision in the head's four threads (same block max, same
      // m_run).  PV(j-1) completed before S(j) (MMAs complete in issue order),
      // so O may be rescaled and P overwritten now.
      const bool need = bm > m_run + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? bm : m_run;
        const float alpha = (m_run == -INFINITY || !need) ? (need ? 0.f : 1.f) : ex2(m_run - m_new);
        if (j > 0 && __any_sync(0xffffffffu, need && m_run != -INFINITY)) {
#pragma unroll 1
          for (int m = 0; m < 2; ++m)
#pragma unroll 1
            for (int cc = 0; cc < 64; cc += 32) {
              const uint32_t oa = tmem + lane_off + kColO + 128 * m + 64 * ch + cc;
              uint32_t o[32];
              tmem_ld32(oa, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(oa, o);
              tmem_st_wait();  // the source registers are reused by the next load
            }
          tc_fence_before();
        }
        l_run *= alpha;
        m_run = m_new;
      }
      const float mu = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float pa = ex2(fmaf(x[2 * i], sl2e, -mu));
        const float pb = ex2(fmaf(x[2 * i + 1], sl2e, -mu));
        l_run += pa + pb;
        pk[i] = pack_bf16x2(pa, pb);
      }
      tc_fence_before();
      {
        // P row hl, slots [64ch + 32half, +32): chunk ch, bytes [64half, 64half+64)
        uint8_t* prow = sm.p[ch] + hl * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(prow + (((4 * half + i) ^ (hl & 7)) << 4)) =
              make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (crank == 0) mbar_arrive(smem_u32(&sm.p_full));
        else mbar_arrive_remote(mapa_shared(smem_u32(&sm.p_full), 0));
      }
    }
    // ------------------------------- epilogue -------------------------------
    bool have = ok && nblk > 0;
    if (have) have = mbar_wait_warp(smem_u32(&sm.mma_done), 0, c, abort_flag);
    tc_fence_after();
    // the head's row sum over its four threads (red[] is free once every warp
    // has passed the first barrier)
    named_bar_sync(1, kSoftWarps * 32);
    sm.red[ws][lane] = l_run;
    named_bar_sync(1, kSoftWarps * 32);
    const float lsum = (sm.red[quad][lane] + sm.red[quad + 4][lane]) +
                       (sm.red[quad ^ 2][lane] + sm.red[(quad ^ 2) + 4][lane]);
    const float inv = (have && lsum > 0.f) ? 1.f / lsum : 0.f;
    __nv_bfloat16* orow = out + (row * kH + kHC * crank + hl) * (long long)kDV;
    const bool all_have = __all_sync(0xffffffffu, have);
#pragma unroll 1
    for (int m = 0; m < 2; ++m)
#pragma unroll 1
      for (int cc = 0; cc < 64; cc += 32) {
        uint32_t o[32];
        if (all_have) {
          tmem_ld32(tmem + lane_off + kColO + 128 * m + 64 * ch + cc, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint4 pk4[4];
        uint32_t* pw = reinterpret_cast<uint32_t*>(pk4);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pw[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + 256 * m + 128 * half + 64 * ch + cc);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = pk4[i];
      }
    if (half == 0 && ch == 0) {
      const long long hrow = row * kH + kHC * crank + hl;
      const bool any = have && m_true != -INFINITY;
      mx[hrow] = any ? m_true * kLn2 : -INFINITY;
      sm_out[hrow] = any ? lsum * ex2(m_run - m_true) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer may still read our shared memory / arrive until here
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc2(tmem, kTmemCols);
  }
}

}  // namespace attn

bool make_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

int attn_fwd_tc_max_topk() { return attn::kMaxTopk; }

int launch_attn_fwd_tc(const Shape& s, const void* q, const void* kv, const int32_t* idx, void* out,
                       float* mx, float* sm, DevCtx c, cudaStream_t st) {
  using namespace attn;
  if (s.topk > kMaxTopk) return DSA_ERR_UNSUPPORTED;
  CUtensorMap tq;
  const uint64_t qrows = (uint64_t)s.B * s.S_q * kH;
  if (!make_tmap_2d_bf16(&tq, q, qrows, kDQK, 64, kHC, 128)) return DSA_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  if (cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long nrows = (long long)s.B * s.S_q;
  attn_fwd_tc_kernel<<<(unsigned)(2 * nrows), kThreads, smem, st>>>(tq, q, kv, s, idx,
                                                                     (__nv_bfloat16*)out, mx, sm,
                                                                     nrows, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
