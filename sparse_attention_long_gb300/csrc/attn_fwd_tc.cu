// Sparse multi-query attention forward on tcgen05 (bf16 in, fp32 accumulate).
//
// [DSA-32K] Sparse Flash Attention forward: p[t] = Softmax(q[t] K_topk^T scale),
// O[t] = p[t] V_topk; the 128 heads of token t share its top-k kv rows, each
// row 576 wide (512 latent + 64 rope) and V = its first 512 columns
// (weight-absorbed MLA).
//
// Persistent CTA pairs (clusters of two), each taking a strided share of the
// query rows; every stage of the pipeline below runs across token
// boundaries, so the next token's indices, query and first kv block load
// while the current one finishes.
//
// Moving the selected kv rows from L2 into shared memory bounds this kernel
// (about 18-24 bytes per cycle per SM through cp.async, whatever the access
// pattern), so each row is gathered once per pair: CTA c gathers its 288
// columns D_c of every selected row, value columns E_c = [128c, 128c+128) u
// [256+128c, 256+128c+128) and rope columns R_c = [512+32c, 512+32c+32).
//
// Every MMA is a two-CTA MMA (cta_group::2, M = 128 = 64 rows per CTA) issued
// by CTA 0.  B is split by N between the CTAs' shared memories, and each
// CTA's accumulator keeps its 64 rows twice over the 128 TMEM lanes: lanes
// 0..63 pair with CTA 0's half of B, lanes 64..127 with CTA 1's half.  With A
// in TMEM, lanes 0..63 and 64..127 of A may hold different data, which splits
// the logit contraction between the CTAs without any exchange.  CTA c owns
// heads [64c, 64c+64).  Per 112-slot block:
//   1. logits (N = 224), 18 steps with A in TMEM: lanes h / 64+h of A hold
//      head h's query columns D_0 / D_1 (value then rope columns); B rows
//      n < 112 are CTA 0's columns D_0 of slot n, rows n >= 112 CTA 1's
//      columns D_1 of slot n - 112.  Lane h of the accumulator ends with head
//      h's partial logit over D_0 for the 112 slots, lane 64+h with the partial
//      over D_1;
//   2. the softmax warps add the two halves through shared memory (the lane
//      pair partner's partials, in two rounds through the P buffer about to be
//      written), take the block max over the head's four threads, run the fp32
//      online softmax (exp2 domain; the running max used for P only moves when
//      a head's block max exceeds it by more than 2^8, so the O rescale in
//      TMEM is rare) and write P as bf16 into shared memory (K-major: row =
//      head, slots contiguous);
//   3. O += P V with N = 256 value columns: B rows n < 128 = CTA 0's value
//      columns, n >= 128 CTA 1's, both from the gathered block (no second
//      gather of V); two MMAs per 16-slot step cover the 512 columns.  O of
//      the CTA's 64 heads takes 256 TMEM columns: O column 128m + i of lane h
//      is value column 256m + i, of lane 64 + h value column 256m + 128 + i.
// TMEM: O 256 + logits 112 + query 144 columns = 512.  Three block stages in
// shared memory (cp.async gathers completing on the stage barrier), two P
// buffers.  The MMA issuer gives the next block's logits priority over a
// ready PV, so the logits of block j+1 run during the softmax of block j.
//
// CTA 0 must know when CTA 1's operands are ready and its logits read.  CTA
// 1's softmax warps signal CTA 0's barriers with 4-byte st.async stores that
// complete on them (a cluster-scope arrive costs the arriving thread ~300
// cycles, the store ~6); CTA 0's first softmax warp expects those bytes when
// it arrives.  CTA 1's gathered blocks reach CTA 0's stage barriers through
// the relay thread (a proxy fence, then a cluster-scope arrive).
//
// Roles per CTA: warp 0 = TMEM allocation, the MMA issuer in CTA 0 and the
// relay in CTA 1; warps 1..4 = kv gather and each token's query columns into
// TMEM (as soon as the previous token's last logits MMA is done, so the
// softmax warps go straight from a token's last block to its epilogue);
// warps 5..12 = softmax and epilogue (warp w: TMEM lane quadrant w % 4, logit
// columns [56ch, 56ch+56) with ch = (w - 5) / 4); warp 13 = index scan of
// the coming tokens (valid-slot masks, block count, out-of-range report) and
// an L2 prefetch of their query rows.
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace attn {

constexpr int kH = 128, kHC = 64, kDQK = 576, kDV = 512;
constexpr int kBlk = 112;                          // slots per block
constexpr int kMaxTopk = 2048;
constexpr int kStages = 3;                         // gathered blocks in shared memory
constexpr int kChunk = kBlk * 128;                 // 112 slots x 64 value columns (SW128 rows)
constexpr int kRope = kBlk * 64;                   // 112 slots x 32 rope columns (SW64 rows)
constexpr int kStageBytes = 4 * kChunk + kRope;
// mask words cover every slot of the last (partial) block, plus one word read
// past it by the funnel shift
constexpr int kMaskWords = (kMaxTopk + kBlk + 63) / 64 + 1;
constexpr int kPBytes = 2 * kHC * 128;             // P: 2 chunks of 64 slots (SW128 rows)
constexpr int kPvSteps = kBlk / 16;                // 16-slot steps of a PV
constexpr int kGatherWarps = 4, kSoftWarps = 8;
constexpr int kSlotsPerWarp = kBlk / kGatherWarps; // 28
constexpr int kWarpGather0 = 1, kWarpSoft0 = kWarpGather0 + kGatherWarps;
constexpr int kWarpScan = kWarpSoft0 + kSoftWarps;
constexpr int kThreads = 32 * (kWarpScan + 1);
constexpr int kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = kColS + kBlk;  // Q: 144 columns
constexpr uint32_t kIdescS = idesc_bf16(128, 2 * kBlk, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);
constexpr float kRescaleThreshold = 8.0f;          // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
static_assert(kColQ + 144 == kTmemCols, "TMEM columns");
static_assert(kChunk % 1024 == 0 && kRope % 512 == 0 && kStageBytes % 1024 == 0, "operand alignment");

struct __align__(1024) Smem {
  uint8_t stage[kStages][kStageBytes];             // [value chunk 0..3 | rope][slot][row]
  uint8_t p[2][kPBytes];                           // P of even / odd blocks (and the exchange)
  unsigned long long mask[2][kMaskWords];          // per token (even / odd): valid slots
  int nblk[2];                                     // per token: blocks up to the last valid slot
  float red[kSoftWarps][32];                       // per-warp partial block maxima / row sums
  uint32_t sink[kSoftWarps];                       // targets of CTA 1's signalling stores
  uint32_t sink_g[kGatherWarps];                   // (those of its gather warps)
  uint64_t st_full[kStages], st_empty[kStages];
  uint64_t s_full, s_free, p_full[2];
  uint64_t q_tm[2], q_free[2], mma_done[2], sc_full[2], sc_empty[2], fin;
  uint32_t tmem_base;
  int abort;
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

__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// bar.red.or over `n` threads of named barrier `id`: true if any thread passed true
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// 4-byte store into the peer CTA's shared memory that completes 4 bytes of the
// transaction count of the peer's barrier `cluster_bar` (release at cluster
// scope); the issuing thread does not wait for it
__device__ __forceinline__ void st_async_signal(uint32_t cluster_addr, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cluster_addr),
               "r"(0u), "r"(cluster_bar)
               : "memory");
}
// hint: bring `bytes` (a multiple of 16) from global memory into L2
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// query columns of one head for one lane half (see the softmax role)
__device__ __forceinline__ const __nv_bfloat16* q_head(const __nv_bfloat16* qb, long long row,
                                                      uint32_t crank, int hl) {
  return qb + (row * kH + kHC * crank + hl) * (long long)kDQK;
}
__device__ __forceinline__ void q_fetch_value(const __nv_bfloat16* qh, int ch, int half, uint32_t (&w0)[32],
                                              uint32_t (&w1)[32]) {
  const uint4* src = reinterpret_cast<const uint4*>(qh + 256 * ch + 128 * half);
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const uint4 a = __ldg(src + t), b = __ldg(src + 8 + t);
    w0[4 * t] = a.x;
    w0[4 * t + 1] = a.y;
    w0[4 * t + 2] = a.z;
    w0[4 * t + 3] = a.w;
    w1[4 * t] = b.x;
    w1[4 * t + 1] = b.y;
    w1[4 * t + 2] = b.z;
    w1[4 * t + 3] = b.w;
  }
}
// ... and into TMEM (lane_tmem = TMEM base with this warp's lane quadrant);
// the rope columns (column half 0 only) are loaded here
__device__ __forceinline__ void q_store(uint32_t lane_tmem, const __nv_bfloat16* qh, int ch, int half,
                                        const uint32_t (&w0)[32], const uint32_t (&w1)[32]) {
  tmem_st32(lane_tmem + kColQ + 64 * ch, w0);
  tmem_st32(lane_tmem + kColQ + 64 * ch + 32, w1);
  if (ch == 0) {
    const uint4* rsrc = reinterpret_cast<const uint4*>(qh + kDV + 32 * half);
    uint32_t w2[16];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 a = __ldg(rsrc + t);
      w2[4 * t] = a.x;
      w2[4 * t + 1] = a.y;
      w2[4 * t + 2] = a.z;
      w2[4 * t + 3] = a.w;
    }
    tmem_st16(lane_tmem + kColQ + 128, w2);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const void* __restrict__ qg, const void* __restrict__ kvg, Shape s,
                       const int32_t* __restrict__ idx, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ mx, float* __restrict__ sm_out, long long nrows,
                       DevCtx c, const __grid_constant__ CUtensorMap tmo) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  // token i of this pair is flattened query row nrows - 1 - (pair + i * npairs):
  // the longest rows of a causal batch first, spread over all pairs
  const long long pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int ntok = pair < nrows ? (int)((nrows - 1 - pair) / npairs + 1) : 0;
  const int k = s.topk;
  volatile int* abort_flag = &sm.abort;
  const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(qg);

  if (threadIdx.x == 32 * kWarpGather0) {
    // CTA 0's barriers that CTA 1's relay also arrives on count one more
    const uint32_t peer = crank == 0 ? 1u : 0u;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.st_full[i]), kGatherWarps * 32 + peer);
      mbar_init(smem_u32(&sm.st_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    // s_free, p_full, q_tm (used in CTA 0): the 8 local softmax warps arrive,
    // the first of them also expecting the 8 x 4 bytes CTA 1's warps store
    mbar_init(smem_u32(&sm.s_free), kSoftWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.p_full[i]), kSoftWarps);  // blocks of parity i
      // tokens of parity i: the local gather warps store the query, the first
      // also expecting CTA 1's gather warps' 4 x 4 bytes (used in CTA 0)
      mbar_init(smem_u32(&sm.q_tm[i]), kGatherWarps);
      mbar_init(smem_u32(&sm.q_free[i]), 1);         // the token's last logits MMA done
      mbar_init(smem_u32(&sm.mma_done[i]), 1);
      mbar_init(smem_u32(&sm.sc_full[i]), 1);
      // the gather warps, the softmax warps and the issuer (CTA 0) / relay (CTA 1)
      mbar_init(smem_u32(&sm.sc_empty[i]), kGatherWarps + kSoftWarps + 1);
    }
    mbar_init(smem_u32(&sm.fin), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  {
    // the block stages start as zeros (slots that are never gathered stay finite)
    uint4* z = reinterpret_cast<uint4*>(&sm.stage[0][0]);
    for (int i = threadIdx.x; i < kStages * kStageBytes / 16; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // generic writes -> the tensor cores' reads
  }
  if (warp == 0) {
    tmem_alloc2(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish2();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kWarpScan) {
    // ------------------------------- index scan -------------------------------
    // Per token: a 64-bit valid-slot mask per 64 slots, the number of blocks up
    // to the last valid slot, and a report of out-of-range entries (skipped).
    // Two tokens in flight (even / odd buffers).
    for (int i = 0; i < ntok; ++i) {
      const int bi = i & 1;
      const long long row = nrows - 1 - (pair + (long long)i * npairs);
      if (lane == 0)  // this CTA's 64 query heads of the token, into L2 ahead of their load
        prefetch_l2_bulk(qb + (row * kH + kHC * crank) * (long long)kDQK, kHC * kDQK * 2);
      if (!mbar_wait_warp(smem_u32(&sm.sc_empty[bi]), ((i >> 1) & 1) ^ 1, c, abort_flag)) break;
      const int32_t* irow = idx + row * (long long)k;
      const int nw = (k + 63) / 64;
      bool bad = false;
      int lastw = -1;
      unsigned long long lastbits = 0;
#pragma unroll 4
      for (int g = 0; g < nw; ++g) {
        const int s0 = 64 * g + lane, s1 = s0 + 32;
        const int i0 = s0 < k ? irow[s0] : -1, i1 = s1 < k ? irow[s1] : -1;
        bad |= (i0 < -1 || i0 >= s.S_k) || (i1 < -1 || i1 >= s.S_k);
        const uint32_t lo = __ballot_sync(0xffffffffu, i0 >= 0 && i0 < s.S_k);
        const uint32_t hi = __ballot_sync(0xffffffffu, i1 >= 0 && i1 < s.S_k);
        const unsigned long long w = ((unsigned long long)hi << 32) | lo;
        if (lane == 0) sm.mask[bi][g] = w;
        if (w) {
          lastw = g;
          lastbits = w;
        }
      }
      for (int g = nw + lane; g < kMaskWords; g += 32) sm.mask[bi][g] = 0ull;
      if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(c, DSA_ERR_INDEX);
      const int last = lastw < 0 ? -1 : 64 * lastw + 63 - __clzll((long long)lastbits);
      if (lane == 0) sm.nblk[bi] = (last + kBlk) / kBlk;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.sc_full[bi]));
    }
  } else if (warp >= kWarpGather0 && warp < kWarpSoft0) {
    // ------------------------------- kv gather -------------------------------
    // Warp gw gathers slots [28gw, 28gw+28) of each block.  Value columns: one
    // warp-wide copy per slot, lanes 0..15 the 256 contiguous bytes of columns
    // [128c, 128c+128), lanes 16..31 those of [256+128c, 256+128c+128), into
    // value chunks 0..3 (SW128 rows).  Rope: 8 slots per copy, 4 lanes per
    // slot, the 64 bytes of columns R_c into the rope chunk (SW64 rows).
    // Invalid slots (past the token's k entries, -1 or out of range) are not
    // copied: they keep an earlier block's row or the zeros the stages start
    // with, so every byte the MMAs read is finite, and their P is 0.  (Copying
    // row 0 for them sent ~80 copies of one row per CTA to the same L2 lines
    // at every token's last block and made that block's gather ~3x slower.)
    const int gw = warp - kWarpGather0;
    const int run = lane >> 4, p16 = lane & 15;
    const int vcol = 256 * run + 128 * (int)crank + 8 * p16;   // this lane's value piece
    const int vchunk = 2 * run + (p16 >> 3), vpc = p16 & 7;
    const int rs = lane >> 2, rp = lane & 3;                   // rope: slot in group of 8, piece
    const int rcol = kDV + 32 * (int)crank + 8 * rp;
    int G = 0;                                                 // blocks so far (all tokens)
    bool ok = true;
    // Token i's query columns of this CTA into TMEM (thread = TMEM lane of
    // this warp's quadrant: head l & 63, lane half l >> 6; value runs ch 0
    // and 1, rope with ch 0), once the previous token's last logits MMA has
    // read the old ones; then one arrive per warp on CTA 0's q_tm (CTA 1's
    // warps: a 4-byte store that completes on it).  Issued after the token's
    // first block of gathers, so both loads are in flight together.
    auto store_q = [&](int i) -> bool {
      if (i > 0) {
        if (!mbar_wait_warp(smem_u32(&sm.q_free[(i - 1) & 1]), ((i - 1) >> 1) & 1, c, abort_flag))
          return false;
        tc_fence_after();
      }
      const int l = (warp & 3) * 32 + lane;
      const long long qrow = nrows - 1 - (pair + (long long)i * npairs);
      const __nv_bfloat16* qh = q_head(qb, qrow, crank, l & 63);
      const uint32_t lane_tmem = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      // 64 value columns at a time (run ch = p >> 1, its half p & 1 -> TMEM
      // columns kColQ + 32p), then the 32 rope columns -> kColQ + 128
      const uint4* vsrc = reinterpret_cast<const uint4*>(qh + 128 * (l >> 6));
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        uint32_t w[32];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint4 a = __ldg(vsrc + 32 * (p >> 1) + 8 * (p & 1) + t);
          w[4 * t] = a.x, w[4 * t + 1] = a.y, w[4 * t + 2] = a.z, w[4 * t + 3] = a.w;
        }
        tmem_st32(lane_tmem + kColQ + 32 * p, w);
        tmem_st_wait();  // w is reused by the next piece
      }
      {
        const uint4* rsrc = reinterpret_cast<const uint4*>(qh + kDV + 32 * (l >> 6));
        uint32_t w2[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 a = __ldg(rsrc + t);
          w2[4 * t] = a.x, w2[4 * t + 1] = a.y, w2[4 * t + 2] = a.z, w2[4 * t + 3] = a.w;
        }
        tmem_st16(lane_tmem + kColQ + 128, w2);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = smem_u32(&sm.q_tm[i & 1]);
        if (crank == 0) {
          if (gw == 0) mbar_arrive_expect_tx(bar, 4 * kGatherWarps);
          else mbar_arrive(bar);
        } else {
          st_async_signal(mapa_shared(smem_u32(&sm.sink_g[gw]), 0), mapa_shared(bar, 0));
        }
      }
      return true;
    };
    for (int i = 0; i < ntok && ok; ++i) {
      const int bi = i & 1;
      if (!mbar_wait_warp(smem_u32(&sm.sc_full[bi]), (i >> 1) & 1, c, abort_flag)) break;
      const int nblk = sm.nblk[bi];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.sc_empty[bi]));
      const long long row = nrows - 1 - (pair + (long long)i * npairs);
      const int32_t* irow = idx + row * (long long)k;
      const __nv_bfloat16* kvb =
          reinterpret_cast<const __nv_bfloat16*>(kvg) + (row / s.S_q) * s.S_k * (long long)kDQK;
      for (int j = 0; j < nblk; ++j, ++G) {
        const int st = G % kStages;
        // this warp's 28 indices of the block (loaded before the wait)
        const int e = j * kBlk + kSlotsPerWarp * gw + lane;
        int id = (lane < kSlotsPerWarp && e < k) ? irow[e] : -1;
        if (id >= s.S_k) id = -1;
        if (!mbar_wait_warp(smem_u32(&sm.st_empty[st]), ((G / kStages) & 1) ^ 1, c, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t base = smem_u32(sm.stage[st]);
#pragma unroll 7
        for (int t = 0; t < kSlotsPerWarp; ++t) {
          const int r = kSlotsPerWarp * gw + t;
          const int rid = __shfl_sync(0xffffffffu, id, t);
          if (rid >= 0)
            cp_async16_cg(base + vchunk * kChunk + r * 128 + ((vpc ^ (r & 7)) << 4),
                          kvb + (long long)rid * kDQK + vcol);
        }
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          const int rl = 8 * g8 + rs;
          const int rid = __shfl_sync(0xffffffffu, id, rl & 31);
          const int r = kSlotsPerWarp * gw + rl;
          if (rl < kSlotsPerWarp && rid >= 0)
            cp_async16_cg(base + 4 * kChunk + r * 64 + ((rp ^ ((r >> 1) & 3)) << 4),
                          kvb + (long long)rid * kDQK + rcol);
        }
        cp_async_arrive_noinc(smem_u32(&sm.st_full[st]));
        if (j == 0 && !store_q(i)) {
          ok = false;
          break;
        }
      }
      if (ok && nblk == 0 && !store_q(i)) ok = false;  // a token with no block still needs its query
    }
    cp_async_wait_all();  // no copy may still be in flight when the CTA exits
  } else if (warp == 0) {
    if (crank == 0 && lane == 0) {
      // ------------------------------- MMA issuer -------------------------------
      // Per token, after its query is in both CTAs' TMEM: issue whichever is
      // ready, the logits S(Gs) first (its gathered block is in, the softmax
      // warps of both CTAs have read S(Gs-1), and the PVs up to block Gs-3
      // are issued: the exchange of block Gs reuses that P buffer only after
      // waiting for PV(Gs-2) itself), else PV(Gp) (both CTAs' P of block Gp
      // written).  A PV goes out whole: splitting it around a logits block
      // measured much slower.  Readiness tests do not block; no progress for
      // the wait budget is a timeout.
      int Gs = 0, Gp = 0;  // blocks so far (all tokens): logits issued / PVs issued
      bool ok = true;
      for (int i = 0; i < ntok && ok; ++i) {
        const int bi = i & 1;
        if (!mbar_wait(smem_u32(&sm.sc_full[bi]), (i >> 1) & 1, c, abort_flag)) break;
        const int nblk = sm.nblk[bi];
        mbar_arrive(smem_u32(&sm.sc_empty[bi]));
        if (!mbar_wait<true>(smem_u32(&sm.q_tm[bi]), (i >> 1) & 1, c, abort_flag)) break;
        tc_fence_after();
        int js = 0, jp = 0;  // this token's S / PV issued
        uint64_t t_idle = 0;
        uint32_t spins = 0;
        while (ok && jp < nblk) {
          bool progressed = false;
          if (js < nblk && js <= jp + 2 &&
              (Gs == 0 || mbar_poll(smem_u32(&sm.s_free), (Gs - 1) & 1)) &&
              mbar_poll(smem_u32(&sm.st_full[Gs % kStages]), (Gs / kStages) & 1)) {
            fence_proxy_async_smem();  // CTA 0's gathered block -> tensor cores (CTA 1's: relay)
            tc_fence_after();
            const uint32_t sb = smem_u32(sm.stage[Gs % kStages]);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma2_ts(tmem + kColS, tmem + kColQ + kk * 8,
                      sdesc(sb + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024, kSw128), kIdescS,
                      kk > 0 ? 1u : 0u);
#pragma unroll
            for (int r = 0; r < 2; ++r)
              mma2_ts(tmem + kColS, tmem + kColQ + 128 + r * 8,
                      sdesc(sb + 4 * kChunk + r * 32, 16, 512, kSw64), kIdescS, 1u);
            commit2(smem_u32(&sm.s_full));
            ++js;
            ++Gs;
            // the token's query columns are free once its last logits are done
            if (js == nblk) commit2(smem_u32(&sm.q_free[bi]));
            progressed = true;
          } else if (jp < js && mbar_poll(smem_u32(&sm.p_full[Gp & 1]), (Gp >> 1) & 1)) {
            tc_fence_after();
            const uint32_t sb = smem_u32(sm.stage[Gp % kStages]), pa = smem_u32(sm.p[Gp & 1]);
#pragma unroll
            for (int kk = 0; kk < kPvSteps; ++kk) {
              const uint64_t ad = sdesc(pa + (kk >> 2) * (kHC * 128) + (kk & 3) * 32, 16, 1024, kSw128);
#pragma unroll
              for (int m = 0; m < 2; ++m)
                mma2_ss(tmem + kColO + 128 * m, ad,
                        sdesc(sb + 2 * m * kChunk + kk * 2048, kChunk, 1024, kSw128), kIdescPV,
                        (jp > 0 || kk > 0) ? 1u : 0u);
            }
            commit2(smem_u32(&sm.st_empty[Gp % kStages]));  // stage and P buffer free on completion
            ++jp;
            ++Gp;
            progressed = true;
          }
          if (progressed) {
            spins = 0;
          } else if ((++spins & 63u) == 0) {  // bounded: no progress for the wait budget
            const uint64_t now = globaltimer();
            if (spins == 64) t_idle = now;
            if (*abort_flag) ok = false;
            else if (now - t_idle > c.budget) {
              set_status(c, DSA_ERR_TIMEOUT);
              *abort_flag = 1;
              ok = false;
            }
          }
        }
        if (ok && nblk == 0) {  // no logits MMA read this query: free it in both CTAs
          mbar_arrive(smem_u32(&sm.q_free[bi]));
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.q_free[bi]), 1));
        }
        commit2(smem_u32(&sm.mma_done[bi]));  // this token's O complete
      }
      commit2(smem_u32(&sm.fin));
      mbar_wait(smem_u32(&sm.fin), 0, c, abort_flag);
    } else if (crank == 1 && lane == 0) {
      // --------------------------- relay (CTA 1 -> CTA 0) ---------------------------
      // Forwards CTA 1's gathered blocks, in order, from CTA 1's stage
      // barriers to CTA 0's (after the proxy fence that makes the cp.async
      // writes visible to the tensor cores).  It learns each token's block
      // count from the scan.
      int tk = 0, nb = 0;                  // tokens read from the scan, their blocks
      int fst = 0;                         // blocks forwarded
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      while (true) {
        bool progressed = false;
        if (tk < ntok && mbar_poll(smem_u32(&sm.sc_full[tk & 1]), (tk >> 1) & 1)) {
          nb += sm.nblk[tk & 1];
          mbar_arrive(smem_u32(&sm.sc_empty[tk & 1]));
          ++tk;
          progressed = true;
        }
        if (fst < nb && mbar_poll(smem_u32(&sm.st_full[fst % kStages]), (fst / kStages) & 1)) {
          fence_proxy_async_smem();  // the gathered block (cp.async writes) -> tensor cores
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.st_full[fst % kStages]), 0));
          ++fst;
          progressed = true;
        }
        if (tk == ntok && fst == nb) break;
        if (progressed) {
          spins = 0;
        } else if ((++spins & 63u) == 0) {
          const uint64_t now = globaltimer();
          if (spins == 64) t_idle = now;
          if (*abort_flag) break;
          if (now - t_idle > c.budget) {
            set_status(c, DSA_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
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
    // Thread (lane l, column half ch) handles slots [56ch, 56ch+56) of head hl:
    // lane half 0 keeps slots [56ch, 56ch+32), lane half 1 [56ch+32, 56ch+56).
    const int kept = half ? 24 : 32;
    const int s0 = 56 * ch + (half ? 32 : 0);           // first kept slot in the block

    // one arrive per warp on CTA 0's barrier `bar` (after __syncwarp): CTA 0's
    // warps arrive, the first also expecting CTA 1's stores; CTA 1's warps
    // store 4 bytes into CTA 0 that complete on that barrier (no wait)
    auto signal = [&](uint64_t* bar) {
      if (lane == 0) {
        if (crank == 0) {
          if (warp == kWarpSoft0) mbar_arrive_expect_tx(smem_u32(bar), 4 * kSoftWarps);
          else mbar_arrive(smem_u32(bar));
        } else {
          st_async_signal(mapa_shared(smem_u32(&sm.sink[ws]), 0), mapa_shared(smem_u32(bar), 0));
        }
      }
    };
    // The 8 softmax warps synchronise with each other through named barriers
    // 1 (bar.sync, 256 threads) and 2 (the per-token vote): every warp
    // executes the same sequence of barriers whatever happens (after a failed
    // wait it keeps going through the token without work, and the vote at the
    // next token makes all of them stop), so they cannot deadlock.
    bool ok = true;
    // the epilogue stages O through the P buffers; one thread stores them
    // with TMA and waits for those reads before the buffers are reused
    const bool o_storer = warp == kWarpSoft0 && lane == 0;
    int G = 0;  // blocks so far (all tokens)
    for (int i = 0; i < ntok; ++i) {
      const int bi = i & 1;
      const long long row = nrows - 1 - (pair + (long long)i * npairs);
      if (o_storer) bulk_wait_read_all();
      if (ok) ok = mbar_wait_warp(smem_u32(&sm.sc_full[bi]), (i >> 1) & 1, c, abort_flag);
      if (named_bar_or(2, kSoftWarps * 32, !ok)) break;
      const int nblk = sm.nblk[bi];
      const unsigned long long* mask = sm.mask[bi];
      float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nblk; ++j, ++G) {
        const int pb = G & 1;
        if (ok) ok = mbar_wait_warp(smem_u32(&sm.s_full), G & 1, c, abort_flag);
        // partial logits of head hl over this lane half's columns
        uint32_t v0[32], v1[16], v2[8];
        if (ok) {
          tc_fence_after();
          const uint32_t sbuf = tmem + lane_off + kColS + 56 * ch;
          tmem_ld32(sbuf, v0);
          tmem_ld16(sbuf + 32, v1);
          tmem_ld8(sbuf + 48, v2);
          tmem_ld_wait(v0);
          tmem_ld_also16(v1);
          tmem_ld_also8(v2);
          tc_fence_before();
          __syncwarp();
          signal(&sm.s_free);  // the logit buffer is free
          // the exchange below reuses P buffer pb, last read by PV(G - 2)
          if (G >= 2)
            ok = mbar_wait_warp(smem_u32(&sm.st_empty[(G - 2) % kStages]), ((G - 2) / kStages) & 1, c,
                                abort_flag);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) v0[t] = 0u;
#pragma unroll
          for (int t = 0; t < 16; ++t) v1[t] = 0u;
#pragma unroll
          for (int t = 0; t < 8; ++t) v2[t] = 0u;
        }
        // Exchange with the lane-pair partner (lane l ^ 64, same ch) through
        // P buffer pb, in two rounds of up to 4 float4 per thread:
        // xb[t][ch][destination half][head].  Half 0 sends slots 32..55 (6
        // float4), half 1 sends slots 0..31 (8 float4).
        float4* xb = reinterpret_cast<float4*>(sm.p[pb]);
        auto xslot = [&](int t, int dest) { return xb + ((t * 2 + ch) * 2 + dest) * kHC + hl; };
        float x[32];                                     // this thread's kept partials, then logits
        if (half == 0) {
#pragma unroll
          for (int t = 0; t < 32; ++t) x[t] = __uint_as_float(v0[t]);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) x[t] = __uint_as_float(v1[t]);
#pragma unroll
          for (int t = 0; t < 8; ++t) x[16 + t] = __uint_as_float(v2[t]);
#pragma unroll
          for (int t = 24; t < 32; ++t) x[t] = 0.f;
        }
#pragma unroll
        for (int rnd = 0; rnd < 2; ++rnd) {
          if (half == 0) {
            // float4 #q of slots 32..55: q = 0..3 from v1, 4..5 from v2
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int q = 4 * rnd + t;
              if (q < 4)
                *xslot(t, 1) = make_float4(__uint_as_float(v1[4 * q]), __uint_as_float(v1[4 * q + 1]),
                                           __uint_as_float(v1[4 * q + 2]), __uint_as_float(v1[4 * q + 3]));
              else if (q < 6)
                *xslot(t, 1) =
                    make_float4(__uint_as_float(v2[4 * (q - 4)]), __uint_as_float(v2[4 * (q - 4) + 1]),
                                __uint_as_float(v2[4 * (q - 4) + 2]), __uint_as_float(v2[4 * (q - 4) + 3]));
            }
          } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int q = 4 * rnd + t;
              *xslot(t, 0) = make_float4(__uint_as_float(v0[4 * q]), __uint_as_float(v0[4 * q + 1]),
                                         __uint_as_float(v0[4 * q + 2]), __uint_as_float(v0[4 * q + 3]));
            }
          }
          named_bar_sync(1, kSoftWarps * 32);
          // receive: the partner's partials for this thread's kept slots
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int q = 4 * rnd + t;
            if (4 * q < kept) {
              const float4 pr = *xslot(t, half);
              x[4 * q] += pr.x;
              x[4 * q + 1] += pr.y;
              x[4 * q + 2] += pr.z;
              x[4 * q + 3] += pr.w;
            }
          }
          named_bar_sync(1, kSoftWarps * 32);            // the region is rewritten next
        }
        // valid slots of the kept range (slot j*kBlk + s0 + t of the token)
        uint32_t vmask;
        {
          const int gs = j * kBlk + s0, w = gs >> 6, sh = gs & 63;
          unsigned long long mk = mask[w] >> sh;
          if (sh) mk |= mask[w + 1] << (64 - sh);
          vmask = (uint32_t)mk & (half ? 0x00ffffffu : 0xffffffffu);
        }
        float bm = -INFINITY;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          if (((vmask >> t) & 1u) == 0) x[t] = -INFINITY;
          bm = fmaxf(bm, x[t]);
        }
        // the head's block max over its four threads (lane pair x column halves)
        sm.red[ws][lane] = bm;
        named_bar_sync(1, kSoftWarps * 32);
        bm = fmaxf(fmaxf(sm.red[quad][lane], sm.red[quad + 4][lane]),
                   fmaxf(sm.red[quad ^ 2][lane], sm.red[(quad ^ 2) + 4][lane]));
        // (red is rewritten only after the next block's first barrier, which
        // every warp reaches only after these reads)
        if (!ok) continue;
        bm *= sl2e;                                        // log2 units (sl2e > 0)
        m_true = fmaxf(m_true, bm);
        // the same decision in the head's four threads (same block max, same m_run)
        const bool need = bm > m_run + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? bm : m_run;
          const float alpha = (m_run == -INFINITY || !need) ? (need ? 0.f : 1.f) : ex2(m_run - m_new);
          if (j > 0 && __any_sync(0xffffffffu, need && m_run != -INFINITY)) {
            // O must hold PV(G-1) before it is rescaled (its completion frees
            // its stage; PV(G) waits for this block's P)
            ok = mbar_wait_warp(smem_u32(&sm.st_empty[(G - 1) % kStages]), ((G - 1) / kStages) & 1, c,
                                abort_flag);
            if (!ok) continue;
            tc_fence_after();
#pragma unroll 1
            for (int m = 0; m < 2; ++m)
#pragma unroll 1
              for (int cc = 0; cc < 64; cc += 32) {
                const uint32_t oa = tmem + lane_off + kColO + 128 * m + 64 * ch + cc;
                uint32_t o[32];
                tmem_ld32(oa, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
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
        for (int t = 0; t < 16; ++t) {
          const float pa = ex2(fmaf(x[2 * t], sl2e, -mu));
          const float pc = ex2(fmaf(x[2 * t + 1], sl2e, -mu));
          l_run += pa + pc;
          pk[t] = pack_bf16x2(pa, pc);
        }
        {
          // P row hl, slots s0 .. s0+kept-1: 16-byte pieces of 8 slots; slot s
          // sits in chunk s / 64, piece (s % 64) / 8 of the head's row
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (8 * q < kept) {
              const int sl = s0 + 8 * q;
              uint8_t* prow = sm.p[pb] + (sl >> 6) * (kHC * 128) + hl * 128;
              *reinterpret_cast<uint4*>(prow + ((((sl & 63) >> 3) ^ (hl & 7)) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        signal(&sm.p_full[pb]);
      }
      // this token's masks are no longer read
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.sc_empty[bi]));
      // ------------------------------- epilogue -------------------------------
      bool have = ok;
      if (have) have = mbar_wait_warp(smem_u32(&sm.mma_done[bi]), (i >> 1) & 1, c, abort_flag);
      ok = have;
      have = have && nblk > 0;
      tc_fence_after();
      // the head's row sum over its four threads
      named_bar_sync(1, kSoftWarps * 32);
      sm.red[ws][lane] = l_run;
      named_bar_sync(1, kSoftWarps * 32);
      const float lsum = (sm.red[quad][lane] + sm.red[quad + 4][lane]) +
                         (sm.red[quad ^ 2][lane] + sm.red[(quad ^ 2) + 4][lane]);
      const float inv = (have && lsum > 0.f) ? 1.f / lsum : 0.f;
      const bool all_have = __all_sync(0xffffffffu, have);
      // O (bf16) out through shared memory, in two rounds m = 0, 1: value
      // columns [256m, 256m+256) of the CTA's 64 heads fill both P buffers
      // (32 KB, free: every PV of this token has completed) as four 64-column
      // tiles [64 heads][128 B] with the 128-byte swizzle, stored by TMA.
      // This thread writes row hl of tile 2*half + ch (value columns 256m +
      // 128half + 64ch .. +64).
      uint8_t* const ostage = &sm.p[0][0];
      uint8_t* const trow = ostage + (2 * half + ch) * (kHC * 128) + hl * 128;
#pragma unroll 1
      for (int m = 0; m < 2; ++m) {
        if (m == 1) {  // round 0's tiles read out of shared memory before they are overwritten
          if (o_storer) bulk_wait_read_all();
          named_bar_sync(1, kSoftWarps * 32);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t o[16];
          if (all_have) {
            tmem_ld16(tmem + lane_off + kColO + 128 * m + 64 * ch + 16 * q4, o);
            tmem_ld_wait16(o);
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) o[t] = 0u;
          }
          uint32_t pw[8];
#pragma unroll
          for (int t = 0; t < 8; ++t)
            pw[t] = pack_bf16x2(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
          *reinterpret_cast<uint4*>(trow + (((2 * q4) ^ (hl & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(trow + (((2 * q4 + 1) ^ (hl & 7)) << 4)) =
              make_uint4(pw[4], pw[5], pw[6], pw[7]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kSoftWarps * 32);
        if (o_storer) {
          const int y = (int)(row * kH + kHC * crank);
#pragma unroll 1
          for (int tt = 0; tt < 4; ++tt) tma_store_2d(&tmo, smem_u32(ostage + tt * (kHC * 128)), 256 * m + 64 * tt, y);
          bulk_commit_group();
        }
      }
      tc_fence_before();  // O is overwritten by the next token's first PV
      if (half == 0 && ch == 0) {
        const long long hrow = row * kH + kHC * crank + hl;
        const bool any = have && m_true != -INFINITY;
        mx[hrow] = any ? m_true * kLn2 : -INFINITY;
        sm_out[hrow] = any ? lsum * ex2(m_run - m_true) : 0.f;
      }
    }
    if (o_storer) bulk_wait_all();
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
  const long long nrows = (long long)s.B * s.S_q;
  if (nrows == 0) return DSA_OK;
  const size_t smem = sizeof(Smem) + 1024;
  if (cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  // persistent: as many CTA pairs as can be resident at once (one CTA per SM)
  static int pairs_by_device[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  int pairs = dev < 64 ? pairs_by_device[dev] : 0;
  if (pairs <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, attn_fwd_tc_kernel, &cfg) != cudaSuccess || clusters <= 0) {
      cudaGetLastError();
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSA_ERR_CUDA;
      clusters = sms / 2;
    }
    pairs = clusters;
    if (dev < 64) pairs_by_device[dev] = pairs;
  }
  if (nrows * kH > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  const long long grid_pairs = nrows < pairs ? nrows : pairs;
  // O stores: [rows * 128 heads][512] bf16 in 64 x 64 tiles, 128-byte swizzle
  CUtensorMap tmo;
  if (!make_tmap_2d_bf16(&tmo, out, (uint64_t)nrows * kH, kDV, 64, kHC, 128)) return DSA_ERR_CUDA;
  attn_fwd_tc_kernel<<<(unsigned)(2 * grid_pairs), kThreads, smem, st>>>(q, kv, s, idx,
                                                                          (__nv_bfloat16*)out, mx, sm,
                                                                          nrows, c, tmo);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
