// Lightning Indexer scores on the 5th-generation tensor cores (bf16, sm_103a).
//
// [DSA-32K] Lightning Indexer forward: I[t,s] = sum_j w[t,j] ReLU(q_I[t,j].k_I[s])
// for the H_I = 64 index heads of token t and one index key per position.
//
// GEMM mapping: one MMA computes D[128 keys x 256] = k_I[128 keys x 128] *
// q_I[4 tokens x 64 heads x 128]^T, so TMEM lane = key and the 64 columns of
// one token hold its 64 heads: the head reduction of the epilogue is
// in-thread (64 ReLU + FMA per score) and each warp stores 32 consecutive
// keys of a token (coalesced).  A CTA owns 4 query rows (B operand resident
// in shared memory, 64 KB) and streams 128-key blocks of k_I through a
// 4-stage TMA ring; two 256-column TMEM accumulators let the epilogue of
// block i overlap the MMA of block i+1.  Only causal blocks are visited and
// only keys s <= pos(t) are stored.
//
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..9 = epilogue (two warps per TMEM lane quadrant, two tokens each).
//
// Fused form (kFused): the scores never leave the SM.  Each token keeps a
// running threshold T in shared memory; after every key block the epilogue
// appends the block's keys whose order-preserving key is >= T to the row's
// candidate list in global memory (value key and position; one warp-wide
// compaction per token and block) and counts them in a 2048-bin histogram of
// the key's upper 11 bits.  T is then raised to the lower edge of the highest
// bin b with (candidates in bins >= b) >= k: at least k candidates are >= T,
// so T never exceeds the row's k-th largest key, every key that can be in
// the top k is kept, and the exact selection runs over the candidates alone
// (topk.cu).  Every candidate admitted while T stood is in a bin >= b, so a
// running count of the candidates in bins >= b is exact.  The four warps of
// a token pair meet at two named barriers around each update (every 8 key
// blocks and after the last one).
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace idxtc {

constexpr int kHI = 64, kDI = 128;
constexpr int kTQ = 4;                    // query rows per CTA tile
constexpr int kN = kTQ * kHI;             // 256: MMA N
constexpr int kBK = 128;                  // keys per block: MMA M
constexpr int kStages = 4;
constexpr int kAChunk = kBK * 128;        // 64 dims x 128 keys, bf16, SW128
constexpr int kAStage = 2 * kAChunk;      // 32 KB
constexpr int kBChunk = kN * 128;         // 32 KB
constexpr int kBBytes = 2 * kBChunk;      // 64 KB
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_bf16(128, kN, false, false);

constexpr int kCandBins = 2048;           // histogram of the key's upper 11 bits

__device__ __forceinline__ uint32_t warp_incl_scan_u32(uint32_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
constexpr int kUpdateEvery = 8;           // key blocks between threshold updates

struct __align__(1024) Smem {
  uint8_t a[kStages][kAStage];
  uint8_t b[kBBytes];
  float w[kTQ][kHI];
  long long pos[kTQ];
  // fused form: per token, bin counts (two 16-bit counts per word), the
  // threshold, the candidates so far, those already counted, the count in
  // bins >= bstar, and the group's abort vote
  uint32_t hist[kTQ][kCandBins / 2];
  uint32_t thr[kTQ], cnt[kTQ], seen[kTQ], cum[kTQ], bstar[kTQ];
  int grp_fail[2];
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], b_full, mma_done;
  uint32_t tmem_base;
  int abort;
  int nkb;
};
static_assert(sizeof(Smem) + 1024 <= 232448, "indexer shared memory");

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      Shape s, const __nv_bfloat16* __restrict__ w, long long row_lo,
                      long long row_hi, long long row_begin, int batch,
                      float* __restrict__ scores, long long ld, uint32_t* __restrict__ cand_key,
                      int32_t* __restrict__ cand_pos, uint32_t* __restrict__ cand_cnt, DevCtx c) {
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
    for (int j = 0; j < kTQ; ++j) sm.thr[j] = sm.cnt[j] = sm.seen[j] = sm.cum[j] = sm.bstar[j] = 0;
    sm.grp_fail[0] = sm.grp_fail[1] = 0;
    fence_mbar_init();
  }
  if (kFused)
    for (int i = threadIdx.x; i < kTQ * kCandBins / 2; i += kThreads) (&sm.hist[0][0])[i] = 0;
  if (threadIdx.x >= 64) {
    const int e = threadIdx.x - 64;  // 256 epilogue threads load w for the 4 rows
    const int j = e / kHI, h = e % kHI;
    const long long row = r0 + j;
    sm.w[j][h] = row < row_hi ? __bfloat162float(w[row * kHI + h]) : 0.f;
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
      tma_load_2d(smem_u32(sm.b) + kBChunk, &tm_q, 64, qrow, bf);
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int st = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        if (!mbar_wait(smem_u32(&sm.empty[st]), ph ^ 1, c, abort_flag)) break;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, kAStage);
        const int krow = (int)((long long)batch * s.S_k + (long long)kb * kBK);
        tma_load_2d(smem_u32(sm.a[st]), &tm_k, 0, krow, fb);
        tma_load_2d(smem_u32(sm.a[st]) + kAChunk, &tm_k, 64, krow, fb);
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
        for (int k = 0; k < kDI / 16; ++k) {
          const uint32_t off = (k & 3) * 32;
          const uint64_t ad = sdesc(a0 + (k >> 2) * kAChunk + off, 16, 1024, kSw128);
          const uint64_t bd = sdesc(b0 + (k >> 2) * kBChunk + off, 16, 1024, kSw128);
          mma_bf16_ss(d, ad, bd, kIdesc, k > 0 ? 1u : 0u);
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
    const int k = s.topk;
    for (int kb = 0; kb < nkb; ++kb) {
      const int acc = kb & 1;
      const bool ok_w = mbar_wait_warp(smem_u32(&sm.acc_full[acc]), (kb >> 1) & 1, c, abort_flag);
      if (!kFused && !ok_w) break;
      if (kFused && !ok_w && lane == 0) sm.grp_fail[half] = 1;  // read at the next update
      tc_fence_after();
      const long long key = (long long)kb * kBK + quad * 32 + lane;
      // both tokens of the warp (2*half, 2*half+1): pipelined TMEM loads
      const int j0 = half * 2;
      const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + acc * kN + j0 * kHI;
      uint32_t A[32], B[32];
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int j = j0 + tt;
        const long long p = sm.pos[j];
        float score = 0.f;
        if (ok_w) score = tt == 0 ? relu_pair_first(tb, sm.w[j0], A, B) : relu_pair_second(tb, sm.w[j], A, B);
        if (!ok_w || p < (long long)kb * kBK) continue;  // whole block masked for this row (warp-uniform)
        if (!kFused) {
          if (key <= p) scores[(r0 + j - row_begin) * ld + key] = score;
        } else if (p >= k) {  // rows with at most k visible keys take all of them: no list
          const uint32_t u = ordered_key(score);
          const bool is_c = key <= p && u >= sm.thr[j];
          const uint32_t bal = __ballot_sync(0xffffffffu, is_c);
          if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&sm.cnt[j], (uint32_t)__popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (is_c) {
              const long long at = (r0 + j - row_begin) * ld + base + __popc(bal & ((1u << lane) - 1u));
              cand_key[at] = u;
              cand_pos[at] = (int32_t)key;
              // one shared atomic per distinct bin of the warp's candidates
              const uint32_t bin = u >> 21;
              const uint32_t peers = __match_any_sync(bal, bin);
              if (lane == __ffs(peers) - 1)
                atomicAdd(&sm.hist[j][bin >> 1], (uint32_t)__popc(peers) << (16 * (bin & 1u)));
            }
          }
        }
      }
      if (kFused && ((kb & (kUpdateEvery - 1)) == kUpdateEvery - 1 || kb == nkb - 1)) {
        // every kUpdateEvery blocks: the group's candidates so far are
        // counted; one warp raises the two tokens' thresholds while the
        // group waits (a warp whose wait failed keeps walking the blocks
        // without work until here, so the group leaves together)
        named_bar_sync(2 + half, 128);
        const bool fail = sm.grp_fail[half] != 0;
        if (!fail && quad == 0) {
          // one warp advances each token's bin pointer 32 bins at a time:
          // past bin b while the candidates in the bins above it still
          // number >= k (cum - prefix >= k, monotone over the lanes)
#pragma unroll 1
          for (int tt = 0; tt < 2; ++tt) {
            const int j = half * 2 + tt;
            if (sm.pos[j] < k) continue;
            const uint32_t total = sm.cnt[j];
            uint32_t cum = sm.cum[j] + (total - sm.seen[j]);
            uint32_t b = sm.bstar[j];
            for (;;) {
              const uint32_t bb = b + lane;
              const uint32_t h = bb < (uint32_t)kCandBins ? (sm.hist[j][bb >> 1] >> (16 * (bb & 1u))) & 0xFFFFu : 0u;
              const uint32_t pre = warp_incl_scan_u32(h, lane);
              const bool adv_ok = bb + 1 < (uint32_t)kCandBins && cum - pre >= (uint32_t)k;
              const int adv = __popc(__ballot_sync(0xffffffffu, adv_ok));
              if (adv > 0) {
                cum -= __shfl_sync(0xffffffffu, pre, adv - 1);
                b += adv;
              }
              if (adv < 32) break;
            }
            if (lane == 0) {
              sm.seen[j] = total;
              sm.cum[j] = cum;
              sm.bstar[j] = b;
              sm.thr[j] = b << 21;
            }
          }
        }
        named_bar_sync(2 + half, 128);
        if (fail) break;
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.acc_empty[acc]));
    }
    if (kFused) {
      named_bar_sync(2 + half, 128);  // the group's last candidates are counted
      if (quad == 0 && lane < 2) {
        const int j = half * 2 + lane;
        if (r0 + j < row_hi) cand_cnt[r0 + j - row_begin] = sm.pos[j] >= k ? sm.cnt[j] : 0u;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace idxtc

// host: 2D bf16 tensor map [rows, cols] with a (box_cols x box_rows) box
bool make_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

namespace idxtc {
template <bool kFused>
static int launch(const Shape& s, const void* q_I, const void* k_I, const void* w, long long row_begin,
                  long long rows, float* scores, long long ld, uint32_t* cand_key,
                  int32_t* cand_pos, uint32_t* cand_cnt, DevCtx c, cudaStream_t st) {
  CUtensorMap tq, tk;
  if (!make_tmap_2d_bf16(&tq, q_I, (uint64_t)s.B * s.S_q * kHI, kDI, 64, kN, 128)) return DSA_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tk, k_I, (uint64_t)s.B * s.S_k, kDI, 64, kBK, 128)) return DSA_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  // per call: the attribute belongs to the current device's context
  if (cudaFuncSetAttribute(indexer_tc_kernel<kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long r_end = row_begin + rows;
  for (int b = 0; b < s.B; ++b) {
    const long long lo = row_begin > (long long)b * s.S_q ? row_begin : (long long)b * s.S_q;
    const long long hi = r_end < (long long)(b + 1) * s.S_q ? r_end : (long long)(b + 1) * s.S_q;
    if (hi <= lo) continue;
    const long long ntiles = (hi - lo + kTQ - 1) / kTQ;
    indexer_tc_kernel<kFused><<<(unsigned)ntiles, kThreads, smem, st>>>(
        tq, tk, s, (const __nv_bfloat16*)w, lo, hi, row_begin, b, scores, ld, cand_key, cand_pos,
        cand_cnt, c);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}
}  // namespace idxtc

int launch_indexer_tc(const Shape& s, const void* q_I, const void* k_I, const void* w,
                      long long row_begin, long long rows, float* scores, long long ld, DevCtx c,
                      cudaStream_t st) {
  return idxtc::launch<false>(s, q_I, k_I, w, row_begin, rows, scores, ld, nullptr, nullptr, nullptr,
                              c, st);
}

// Fused indexer + candidate filter: for rows [row_begin, row_begin + rows),
// row r's candidates (order-preserving keys, positions) go to
// cand_key / cand_pos [(r - row_begin) * ld ...] and their number to
// cand_cnt[r - row_begin] (0 for rows with at most k visible keys).
// ld >= S_k; S_k < 65536 (16-bit bin counts).
int launch_indexer_topk_tc(const Shape& s, const void* q_I, const void* k_I, const void* w,
                           long long row_begin, long long rows, uint32_t* cand_key, int32_t* cand_pos,
                           uint32_t* cand_cnt, long long ld, DevCtx c, cudaStream_t st) {
  if (s.S_k >= 65536 || ld < s.S_k) return DSA_ERR_UNSUPPORTED;
  return idxtc::launch<true>(s, q_I, k_I, w, row_begin, rows, nullptr, ld, cand_key, cand_pos, cand_cnt,
                             c, st);
}

}  // namespace dsa
