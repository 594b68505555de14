// Per-query top-k over the indexer scores (exact, bit-reproducible).
//
// [DSA-32K] "Top-k positions of each token" select the kv rows the sparse
// attention gathers.  Order key: value descending, then index ascending;
// -0.0 == +0.0.  Output in ascending index order, -1 padded when fewer than k
// keys are visible.
//
// One CTA of 1024 threads per query row.  The row's n = pos+1 fp32 scores are
// read once (coalesced float4) and held in registers; an MSB-first radix
// select (12 + 12 + 8 bits of the order-preserving key) finds the k-th key T
// and how many keys equal to T are taken; one block-wide scan over the row in
// index order then writes the winners already sorted.  Rows longer than the
// register capacity (4096 * VEC) take the streaming variant, which re-reads
// the row from global memory on every pass.
#include "dsa_common.cuh"

namespace dsa {

constexpr int TK_THREADS = 1024;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_HIST = 4096;

struct TopkSmem {
  uint32_t hist[TK_HIST];
  uint32_t warp_sum[TK_WARPS];
  unsigned long long warp_sum64[TK_WARPS];
  uint32_t total;
  unsigned long long total64;
  uint32_t bin, above, bin_count;
};

// Exclusive scan of v over the 1024 threads in threadIdx order; `total` gets
// the block sum.  Uses sm.warp_sum / sm.total; ends synced (smem reusable).
template <typename U>
__device__ __forceinline__ U block_scan_excl(U v, U* ws, U* s_total, U& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  U x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    U y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const U s = ws[lane];
    U t = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      U y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    ws[lane] = t - s;
    if (lane == 31) *s_total = t;
  }
  __syncthreads();
  const U r = ws[warp] + x - v;
  total = *s_total;
  __syncthreads();
  return r;
}

// Given hist[0..nbins) and k_rem, find the bin b (scanning from the top) with
// count(>b) < k_rem <= count(>=b).  Result in sm.bin / sm.above / sm.bin_count.
__device__ __forceinline__ void find_bin(TopkSmem& sm, int nbins, uint32_t k_rem) {
  if (threadIdx.x == 0) {  // defined result even if no bin qualifies
    sm.bin = 0;
    sm.above = 0;
    sm.bin_count = 0;
  }
  const int per = nbins / TK_THREADS > 0 ? nbins / TK_THREADS : 1;
  const int groups = nbins / per;
  const int i = threadIdx.x;
  uint32_t local = 0;
  const int hi = nbins - i * per;  // this thread covers bins [hi-per, hi)
  if (i < groups)
    for (int b = hi - 1; b >= hi - per; --b) local += sm.hist[b];
  uint32_t total;
  uint32_t excl = block_scan_excl<uint32_t>(local, sm.warp_sum, &sm.total, total);
  if (i < groups && excl < k_rem && excl + local >= k_rem) {
    uint32_t acc = excl;
    for (int b = hi - 1; b >= hi - per; --b) {
      uint32_t h = sm.hist[b];
      if (acc + h >= k_rem) {
        sm.bin = b;
        sm.above = acc;
        sm.bin_count = h;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

// A row with n <= k visible keys takes all of them: out = 0, 1, ..., n-1,
// then -1 (16-byte stores when the row allows them).
__device__ __forceinline__ void write_prefix_rows(int32_t* out, int n, int k, int nt, int tid) {
  if ((k & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
    for (int j = tid; j < k / 4; j += nt) {
      const int b = 4 * j;
      const int4 v = make_int4(b < n ? b : -1, b + 1 < n ? b + 1 : -1, b + 2 < n ? b + 2 : -1,
                               b + 3 < n ? b + 3 : -1);
      reinterpret_cast<int4*>(out)[j] = v;
    }
    return;
  }
  for (int j = tid; j < k; j += nt) out[j] = j < n ? j : -1;
}

// Radix passes shared by both variants.  KEYS(fn) must call fn(key) for every
// valid element of the row.  Returns (via refs) the shift sh of the deepest
// pass, the threshold prefix Tp = T >> sh and the number `take_eq` of
// elements with key>>sh == Tp to keep (lowest indices first).
template <typename ForEach>
__device__ __forceinline__ void radix_select(TopkSmem& sm, int k, ForEach for_each, int& sh_out,
                                             uint32_t& tp_out, uint32_t& take_eq) {
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  uint32_t prefix = 0, pmask = 0, k_rem = (uint32_t)k;
  int sh = 32;
  for (int p = 0; p < 3; ++p) {
    const int s = shifts[p], nb = 1 << widths[p];
    for (int b = threadIdx.x; b < nb; b += TK_THREADS) sm.hist[b] = 0;
    __syncthreads();
    for_each([&](uint32_t key) {
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> s) & (nb - 1)], 1u);
    });
    __syncthreads();
    find_bin(sm, nb, k_rem);
    const uint32_t b = sm.bin, cnt = sm.bin_count;
    k_rem -= sm.above;
    prefix |= b << s;
    pmask |= (uint32_t)(nb - 1) << s;
    sh = s;
    __syncthreads();
    if (cnt == k_rem) break;  // every element of this bin is taken
  }
  sh_out = sh;
  tp_out = prefix >> sh;
  take_eq = k_rem;
}

// Register-resident variant: thread t holds the KPT consecutive scores
// [t*KPT, t*KPT + KPT) of the row (positions past the row end read as key 0
// and are masked out), so one block scan of per-thread counts gives every
// winner its output slot in index order.  The later radix passes only touch
// the keys whose prefix matched the previous pass; each pass has its own
// histogram, all cleared at the start, and the threshold search takes two
// barriers.
constexpr int TK_CAND = 4096;
template <int CAND>
struct __align__(16) TopkRegSmemT {
  uint32_t hist[2 * TK_HIST + 256];  // pass 1 | pass 2 | pass 3
  uint32_t cand[CAND];               // keys of the threshold's pass-1 bin
  uint32_t ws[TK_WARPS];
  uint32_t bin, above, bin_count;
  uint32_t n_cand;  // candidate slots handed out so far (this row)
  int abort_flag;
  unsigned long long bar;  // stage-full barrier (8-byte aligned by the layout)
};

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// A block runs GROUPS independent rows at a time, one per group of GT
// consecutive threads; a group synchronises on named barrier 1 + grp (the
// whole block's barrier when there is one group).
template <int GROUPS, int GT>
__device__ __forceinline__ void gsync(int grp) {
  if constexpr (GROUPS == 1) {
    __syncthreads();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(GT) : "memory");
  }
}
template <int GROUPS, int GT>
__device__ __forceinline__ bool gsync_or(int grp, bool v) {
  if constexpr (GROUPS == 1) {
    return __syncthreads_or(v) != 0;
  } else {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(1 + grp), "r"(GT)
        : "memory");
    return r != 0;
  }
}

// Exclusive scan of v over the GT threads of the group in thread order (tid =
// index in the group); one barrier.  ws must not be written again before the
// next barrier every thread of the group passes.
template <int GT, int GROUPS>
__device__ __forceinline__ uint32_t group_excl_scan_1b(uint32_t v, uint32_t* ws, int tid, int grp) {
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t x = warp_incl_scan(v, lane);
  if (lane == 31) ws[warp] = x;
  gsync<GROUPS, GT>(grp);
  const uint32_t t = lane < GT / 32 ? ws[lane] : 0u;
  const uint32_t ti = warp_incl_scan(t, lane);
  return __shfl_sync(0xffffffffu, ti - t, warp) + x - v;
}

// The bin b of hist[0..NB), counted from the top, with
// count(> b) < k_rem <= count(>= b); result in sm.bin / above / bin_count.
template <int NB, int GT, int GROUPS, typename SM>
__device__ __forceinline__ void find_bin_2b(SM& sm, const uint32_t* hist, uint32_t k_rem, int tid,
                                            int grp) {
  constexpr int PER = NB >= GT ? NB / GT : 1;
  static_assert(PER == 1 || PER % 4 == 0, "bins per thread");
  const int lane = tid & 31, warp = tid >> 5;
  const int hi = NB - tid * PER;  // this thread: bins [hi-PER, hi)
  uint32_t local = 0;
  if constexpr (PER >= 4) {
#pragma unroll
    for (int u = 0; u < PER / 4; ++u) {
      const uint4 v = *reinterpret_cast<const uint4*>(hist + hi - PER + 4 * u);
      local += (v.x + v.y) + (v.z + v.w);
    }
  } else {
    local = hi > 0 ? hist[hi - 1] : 0u;
  }
  const uint32_t x = warp_incl_scan(local, lane);
  if (lane == 31) sm.ws[warp] = x;
  if (tid == 0) sm.bin = 0, sm.above = 0, sm.bin_count = 0;
  gsync<GROUPS, GT>(grp);
  const uint32_t t = lane < GT / 32 ? sm.ws[lane] : 0u;
  const uint32_t ti = warp_incl_scan(t, lane);
  uint32_t acc = __shfl_sync(0xffffffffu, ti - t, warp) + x - local;
  if (acc < k_rem && acc + local >= k_rem) {  // the one thread whose bins hold it
    for (int j = 0; j < PER && hi - 1 - j >= 0; ++j) {
      const uint32_t h = hist[hi - 1 - j];
      if (acc + h >= k_rem) {
        sm.bin = (uint32_t)(hi - 1 - j);
        sm.above = acc;
        sm.bin_count = h;
        break;
      }
      acc += h;
    }
  }
  gsync<GROUPS, GT>(grp);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// (mask << 1) | (a > b), given nb = ~b: a + ~b carries out exactly when a > b.
__device__ __forceinline__ uint32_t shift_in_gt(uint32_t mask, uint32_t a, uint32_t nb) {
  uint32_t r;
  asm("{\n .reg .u32 t;\n add.cc.u32 t, %1, %2;\n addc.u32 %0, %3, %3;\n}"
      : "=r"(r)
      : "r"(a), "r"(nb), "r"(mask));
  return r;
}

// Persistent: a CTA takes GROUPS rows at a time, one per group of GT = NT /
// GROUPS threads (group grp of CTA b: rows GROUPS*b + grp, then + GROUPS *
// gridDim.x, ...); two groups let one row's barrier phases overlap the
// other's work.  When the scores are reachable by TMA (tma_elems > 0: the
// first tma_elems columns of every row, viewed as 128-byte lines) one thread
// of a group loads its next row into the group's shared-memory stage as soon
// as the current one has been read from it, so the next row streams in while
// this one is selected.  The 128-byte swizzle puts 16-byte piece g of a row
// at g ^ ((g >> 3) & 7), so the 8 lanes of a quarter-warp reading their
// consecutive pieces hit distinct banks.
template <int KPT, int NT, int GROUPS>
__global__ void __launch_bounds__(NT, TK_THREADS / NT)
    topk_reg_kernel(const __grid_constant__ CUtensorMap tm, Shape s, const float* __restrict__ scores,
                    long long ld, long long row_begin, long long rows, int32_t* __restrict__ idx,
                    DevCtx c, int tma_elems) {
  static_assert(KPT % 4 == 0 && KPT <= 32, "keys per thread");
  constexpr int GT = NT / GROUPS;                     // threads per row
  constexpr int CAND = GROUPS == 1 ? TK_CAND : TK_CAND / 2;
  using Smem = TopkRegSmemT<CAND>;
  constexpr int C = KPT / 4;                          // 16-byte pieces per thread
  constexpr int BOX_ROWS = 32 * KPT < 256 ? 32 * KPT : 256;  // 128-byte lines per TMA box
  constexpr int BOX_ELEMS = BOX_ROWS * 32;
  extern __shared__ uint8_t dyn_smem[];  // [align 1024] stage per group | Smem per group
  const uint32_t base = smem_u32(dyn_smem);
  uint8_t* aligned = dyn_smem + (((base + 1023u) & ~1023u) - base);
  const int grp = GROUPS == 1 ? 0 : (int)threadIdx.x / GT;
  const int tid = (int)threadIdx.x - grp * GT;        // thread index in the group
  // the row stages exist only in the 1024-thread forms (the others load
  // directly: two to four of them share an SM)
  constexpr int STAGE_BYTES = NT == TK_THREADS ? GT * KPT * 4 : 0;
  const float4* stage = reinterpret_cast<const float4*>(aligned + grp * STAGE_BYTES);
  Smem& sm = reinterpret_cast<Smem*>(aligned + GROUPS * STAGE_BYTES)[grp];
  volatile int* abort_flag = &sm.abort_flag;
  const uint32_t bar = smem_u32(&sm.bar), stage_u32 = smem_u32(aligned + grp * STAGE_BYTES);
  const int k = s.topk;
  // winners staged in shared memory and written as 16-byte pieces (every
  // row's output 16-byte aligned), in the forms that run several CTAs per SM:
  // with one CTA per SM the extra barrier costs more than the scattered
  // stores (measured per wave: 256 threads -4 us, 1024 threads +6-8 us)
  const bool stage_out = GROUPS == 1 && NT < TK_THREADS && k <= CAND && (k & 3) == 0 &&
                         (reinterpret_cast<uintptr_t>(idx) & 15u) == 0;
  const int e0 = tid * KPT;  // this thread's first element of a row
  const bool staged = tma_elems > 0 && e0 + KPT <= tma_elems;  // my keys come from the stage
  // 32-bit row -> position arithmetic when it fits (a 64-bit modulo is slow)
  const bool narrow = s.q_row_index == nullptr && row_begin + rows <= 0x7FFFFFFFll;
  auto row_len = [&](long long rl) -> long long {  // n = pos + 1, or -1 for a bad position
    const long long pos =
        narrow ? s.q_row_offset + (long long)((uint32_t)(row_begin + rl) % (uint32_t)s.S_q)
               : row_pos(s, row_begin + rl);
    return (pos < 0 || pos >= s.S_k) ? -1 : pos + 1;
  };
  auto loads_row = [&](long long rl) { return tma_elems > 0 && rl < rows && row_len(rl) > k; };
  // The block's last thread stages rows: it holds no keys of rows shorter
  // than NT * KPT - KPT and no pass-2 candidate while the threshold's bin
  // holds fewer than NT keys, so the copy is issued off the barrier chain.
  auto issue = [&](long long rl) {  // stage row rl if it is selected from
    if (tid != GT - 1 || !loads_row(rl)) return;
    const int nn = (int)row_len(rl);
    const int nbox = (min(nn, tma_elems) + BOX_ELEMS - 1) / BOX_ELEMS;
    fence_proxy_async_smem();  // the stage's earlier reads come before these writes
    mbar_arrive_expect_tx(bar, (uint32_t)(nbox * BOX_ELEMS * 4));
    for (int bx = 0; bx < nbox; ++bx)
      tma_load_3d(stage_u32 + bx * BOX_ELEMS * 4, &tm, 0, bx * BOX_ROWS, (int)rl, bar);
  };
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  const long long first = (long long)blockIdx.x * GROUPS + grp, step = (long long)gridDim.x * GROUPS;
  issue(first);
  for (long long rl = first; rl < rows; rl += step) {
    int32_t* out = idx + rl * (long long)k;
    const long long nl = row_len(rl);
    if (nl < 0) {
      if (tid == 0) set_status(c, DSA_ERR_INDEX);
      write_prefix_rows(out, 0, k, GT, tid);
      issue(rl + step);
      continue;
    }
    if (nl <= k) {
      write_prefix_rows(out, (int)nl, k, GT, tid);
      issue(rl + step);
      continue;
    }
    const int n = (int)nl;
    const int nv = min(max(n - e0, 0), KPT);
    const uint32_t vmask = nv >= 32 ? 0xFFFFFFFFu : ((1u << nv) - 1u);
    const float* src = scores + rl * ld;
    uint32_t key[KPT];
    bool ok = true;
    if (tma_elems > 0) {
      ok = mbar_wait(bar, phase, c, abort_flag);
      phase ^= 1u;
    }
    if (staged) {
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const int g = tid * C + j;
        const float4 v = stage[g ^ ((g >> 3) & 7)];
        key[4 * j] = ordered_key(v.x);
        key[4 * j + 1] = ordered_key(v.y);
        key[4 * j + 2] = ordered_key(v.z);
        key[4 * j + 3] = ordered_key(v.w);
      }
      if (nv < KPT) {
#pragma unroll
        for (int q = 0; q < KPT; ++q)
          if (q >= nv) key[q] = 0u;
      }
    } else {
#pragma unroll
      for (int q = 0; q < KPT; ++q) key[q] = q < nv ? ordered_key(__ldcs(src + e0 + q)) : 0u;
    }
    for (int i = tid; i < 2 * TK_HIST + 256; i += GT) sm.hist[i] = 0;
    if (tid == 0) sm.n_cand = 0;
    if (gsync_or<GROUPS, GT>(grp, !ok)) return;  // a stage load that never landed: give up
    // pass 1: bits 31..20 of every key
    uint32_t* h1 = sm.hist;
    if (nv == KPT) {
#pragma unroll
      for (int q = 0; q < KPT; ++q) atomicAdd(&h1[key[q] >> 20], 1u);
    } else {
#pragma unroll
      for (int q = 0; q < KPT; ++q)
        if (q < nv) atomicAdd(&h1[key[q] >> 20], 1u);
    }
    gsync<GROUPS, GT>(grp);
    find_bin_2b<TK_HIST, GT, GROUPS>(sm, h1, (uint32_t)k, tid, grp);
    uint32_t k_rem = (uint32_t)k - sm.above;
    const uint32_t b1 = sm.bin, c1 = sm.bin_count;
    // keys above bin b1 (all taken) and keys in it, as bit masks over q
    const uint32_t lo1 = b1 << 20, hi1 = lo1 | 0xFFFFFu;
    uint32_t gtm = 0, eqm = 0;  // shifted in from q = 0 (ends in bit KPT-1), reversed below
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      gtm = shift_in_gt(gtm, key[q], ~hi1);
      eqm = shift_in_gt(eqm, key[q], ~(lo1 - 1u));  // key >= lo1 (when lo1 > 0)
    }
    if (lo1 == 0) eqm = 0xFFFFFFFFu;
    gtm = (__brev(gtm) >> (32 - KPT)) & vmask;
    eqm = (__brev(eqm) >> (32 - KPT)) & ~gtm & vmask;
    if (c1 != k_rem && c1 <= (uint32_t)CAND) {
      // the c1 keys of bin b1 go to shared memory and the later passes run
      // over them alone; each thread's keys take consecutive slots (one
      // shared counter bumped once per warp), the order across threads is
      // immaterial: the passes only count them, and each thread re-reads its
      // own to classify them
      const int lane = threadIdx.x & 31;
      const uint32_t mine = (uint32_t)__popc(eqm);
      const uint32_t incl = warp_incl_scan(mine, lane);
      uint32_t wbase = 0;
      if (lane == 31 && incl > 0) wbase = atomicAdd(&sm.n_cand, incl);
      uint32_t off = __shfl_sync(0xffffffffu, wbase, 31) + incl - mine;
      for (uint32_t m = eqm; m; m &= m - 1u) {
        const int q = __ffs(m) - 1;
        const int g = tid * C + (q >> 2);
        const float v = staged ? reinterpret_cast<const float*>(stage + (g ^ ((g >> 3) & 7)))[q & 3]
                               : src[e0 + q];
        sm.cand[off++] = ordered_key(v);
      }
      gsync<GROUPS, GT>(grp);  // candidates complete; the stage is free
      issue(rl + step);
      uint32_t* h2 = sm.hist + TK_HIST;
      for (uint32_t i = tid; i < c1; i += GT)
        atomicAdd(&h2[(sm.cand[i] >> 8) & 0xFFFu], 1u);
      gsync<GROUPS, GT>(grp);
      find_bin_2b<TK_HIST, GT, GROUPS>(sm, h2, k_rem, tid, grp);
      k_rem -= sm.above;
      uint32_t tp = (b1 << 12) | sm.bin;
      int sh = 8;
      if (sm.bin_count != k_rem) {
        uint32_t* h3 = sm.hist + 2 * TK_HIST;
        const uint32_t b2 = sm.bin;
        for (uint32_t i = tid; i < c1; i += GT) {
          const uint32_t kk = sm.cand[i];
          if (((kk >> 8) & 0xFFFu) == b2) atomicAdd(&h3[kk & 0xFFu], 1u);
        }
        gsync<GROUPS, GT>(grp);
        find_bin_2b<256, GT, GROUPS>(sm, h3, k_rem, tid, grp);
        k_rem -= sm.above;
        sh = 0;
        tp = (tp << 8) | sm.bin;
      }
      // classify this thread's candidates against the final threshold
      const uint32_t tmin = tp << sh, tmax = tmin | ((1u << sh) - 1u);
      uint32_t i = off - (uint32_t)__popc(eqm), cgt = 0, ceq = 0;
      for (uint32_t m = eqm; m; m &= m - 1u, ++i) {
        const uint32_t kk = sm.cand[i], bit = m & (0u - m);
        if (kk > tmax)
          cgt |= bit;
        else if (kk >= tmin)
          ceq |= bit;
      }
      gtm |= cgt;
      eqm = ceq;
    } else if (c1 != k_rem) {
      // more than CAND keys share the bin (heavy ties): passes over registers
      issue(rl + step);
      uint32_t tp = b1;
      int sh = 20;
      uint32_t* h2 = sm.hist + TK_HIST;
#pragma unroll
      for (int q = 0; q < KPT; ++q)
        if (q < nv && key[q] - lo1 < (1u << 20)) atomicAdd(&h2[(key[q] >> 8) & 0xFFFu], 1u);
      gsync<GROUPS, GT>(grp);
      find_bin_2b<TK_HIST, GT, GROUPS>(sm, h2, k_rem, tid, grp);
      k_rem -= sm.above;
      sh = 8;
      tp = (tp << 12) | sm.bin;
      if (sm.bin_count != k_rem) {
        uint32_t* h3 = sm.hist + 2 * TK_HIST;
        const uint32_t lo2 = tp << 8;
#pragma unroll
        for (int q = 0; q < KPT; ++q)
          if (q < nv && key[q] - lo2 < 256u) atomicAdd(&h3[key[q] & 0xFFu], 1u);
        gsync<GROUPS, GT>(grp);
        find_bin_2b<256, GT, GROUPS>(sm, h3, k_rem, tid, grp);
        k_rem -= sm.above;
        sh = 0;
        tp = (tp << 8) | sm.bin;
      }
      const uint32_t tmin = tp << sh, tmax = tmin | ((1u << sh) - 1u);
      uint32_t cgt = 0, ceq = 0;
#pragma unroll
      for (int q = 0; q < KPT; ++q) {
        cgt |= (key[q] > tmax ? 1u : 0u) << q;
        ceq |= (key[q] >= tmin ? 1u : 0u) << q;
      }
      gtm = cgt & vmask;
      eqm = ceq & ~cgt & vmask;
    } else {
      issue(rl + step);  // every key of bin b1 is taken
    }
    const uint32_t take_eq = k_rem;
    const uint32_t p = group_excl_scan_1b<GT, GROUPS>(
        (uint32_t)__popc(gtm) | ((uint32_t)__popc(eqm) << 16), sm.ws, tid, grp);
    uint32_t gt_b = p & 0xFFFFu, eq_b = p >> 16;
    // exactly k winners: they are placed in the candidate list (free once the
    // scan's barrier is passed: every thread has classified its candidates)
    // and leave in 16-byte stores, rather than as scattered 4-byte stores
    int32_t* dst = stage_out ? reinterpret_cast<int32_t*>(sm.cand) : out;
    for (uint32_t m = gtm | eqm; m; m &= m - 1u) {
      const int q = __ffs(m) - 1;
      if ((gtm >> q) & 1u) {
        const uint32_t o = gt_b + min(eq_b, take_eq);
        if (o < (uint32_t)k) dst[o] = e0 + q;
        ++gt_b;
      } else {
        if (eq_b < take_eq && gt_b + eq_b < (uint32_t)k) dst[gt_b + eq_b] = e0 + q;
        ++eq_b;
      }
    }
    if (stage_out) {
      gsync<GROUPS, GT>(grp);
      const int4* sv = reinterpret_cast<const int4*>(sm.cand);
      int4* ov = reinterpret_cast<int4*>(out);
      for (int i = tid; i < k / 4; i += GT) ov[i] = sv[i];
    }
  }
}

// Streaming variant for rows longer than the register capacity: each pass
// re-reads the row (L2 / HBM); compaction walks the row in 4096-element tiles.
__global__ void __launch_bounds__(TK_THREADS, 1)
    topk_stream_kernel(Shape s, const float* __restrict__ scores, long long ld,
                       long long row_begin, int32_t* __restrict__ idx, DevCtx c) {
  __shared__ TopkSmem sm;
  const long long r_local = blockIdx.x;
  const long long row = row_begin + r_local;
  const int k = s.topk;
  int32_t* out = idx + r_local * (long long)k;
  const long long pos = row_pos(s, row);
  if (pos < 0 || pos >= s.S_k) {
    if (threadIdx.x == 0) set_status(c, DSA_ERR_INDEX);
    write_prefix_rows(out, 0, k, TK_THREADS, threadIdx.x);
    return;
  }
  const int n = (int)pos + 1;
  if (n <= k) {
    write_prefix_rows(out, n, k, TK_THREADS, threadIdx.x);
    return;
  }
  const float* src = scores + r_local * ld;
  auto for_each = [&](auto fn) {
    for (int e = threadIdx.x; e < n; e += TK_THREADS) fn(ordered_key(src[e]));
  };
  int sh;
  uint32_t tp, take_eq;
  radix_select(sm, k, for_each, sh, tp, take_eq);
  unsigned long long base = 0;  // packed (gt | eq << 32) counts of earlier tiles
  for (int t0 = 0; t0 < n; t0 += TK_THREADS * 4) {
    const int e0 = t0 + threadIdx.x * 4;
    uint32_t kk[4];
    unsigned long long cnt = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      kk[q] = (e0 + q < n) ? (ordered_key(src[e0 + q]) >> sh) : 0u;
      if (e0 + q < n) cnt += (kk[q] > tp) ? 1ull : ((kk[q] == tp) ? (1ull << 32) : 0ull);
    }
    unsigned long long total;
    unsigned long long p =
        base + block_scan_excl<unsigned long long>(cnt, sm.warp_sum64, &sm.total64, total);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e0 + q < n) {
        const unsigned long long gt_b = p & 0xFFFFFFFFull, eq_b = p >> 32;
        if (kk[q] > tp) {
          const unsigned long long o = gt_b + min(eq_b, (unsigned long long)take_eq);
          if (o < (unsigned long long)k) out[o] = e0 + q;
          p += 1ull;
        } else if (kk[q] == tp) {
          if (eq_b < take_eq && gt_b + eq_b < (unsigned long long)k) out[gt_b + eq_b] = e0 + q;
          p += 1ull << 32;
        }
      }
    }
    base += total;
  }
}

// Exact top-k over the candidates the fused indexer kept for each row
// (indexer_tc.cu, kFused): every key that can be among the row's k largest is
// a candidate, so the radix select over the candidates' keys finds the row's
// threshold.  Candidates arrive in no particular order; they are marked in
// two position bitmaps (above the threshold / equal to it) and one scan over
// the bitmaps in position order writes the winners sorted, the lowest
// positions among equal keys first.  One CTA per row.
__global__ void __launch_bounds__(TK_THREADS, 1)
    topk_cand_kernel(Shape s, const uint32_t* __restrict__ cand_key,
                     const int32_t* __restrict__ cand_pos, const uint32_t* __restrict__ cand_cnt,
                     long long ld, long long row_begin, int32_t* __restrict__ idx, DevCtx c) {
  __shared__ TopkSmem sm;
  extern __shared__ uint32_t marks[];  // [nw] above the threshold | [nw] equal to it
  const long long r_local = blockIdx.x;
  const long long row = row_begin + r_local;
  const int k = s.topk;
  int32_t* out = idx + r_local * (long long)k;
  const long long pos = row_pos(s, row);
  if (pos < 0 || pos >= s.S_k) {
    if (threadIdx.x == 0) set_status(c, DSA_ERR_INDEX);
    write_prefix_rows(out, 0, k, TK_THREADS, threadIdx.x);
    return;
  }
  const int n = (int)pos + 1;
  if (n <= k) {
    write_prefix_rows(out, n, k, TK_THREADS, threadIdx.x);
    return;
  }
  const uint32_t m = cand_cnt[r_local] < (uint32_t)n ? cand_cnt[r_local] : (uint32_t)n;
  const uint32_t* ck = cand_key + r_local * ld;
  const int32_t* cp = cand_pos + r_local * ld;
  auto for_each = [&](auto fn) {
    for (uint32_t i = threadIdx.x; i < m; i += TK_THREADS) fn(ck[i]);
  };
  int sh;
  uint32_t tp, take_eq;
  radix_select(sm, k, for_each, sh, tp, take_eq);
  const int nw = (n + 31) >> 5;
  uint32_t* gtb = marks;
  uint32_t* eqb = marks + nw;
  for (int i = threadIdx.x; i < 2 * nw; i += TK_THREADS) marks[i] = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < m; i += TK_THREADS) {
    const uint32_t kk = ck[i] >> sh;
    const int p = cp[i];
    if (p < 0 || p >= n) continue;
    if (kk > tp)
      atomicOr(&gtb[p >> 5], 1u << (p & 31));
    else if (kk == tp)
      atomicOr(&eqb[p >> 5], 1u << (p & 31));
  }
  __syncthreads();
  // thread t scans the words [t * wpt, t * wpt + wpt), in position order
  const int wpt = (nw + TK_THREADS - 1) / TK_THREADS;
  const int w0 = threadIdx.x * wpt;
  unsigned long long cnt = 0;
  for (int i = 0; i < wpt; ++i)
    if (w0 + i < nw)
      cnt += (unsigned long long)__popc(gtb[w0 + i]) | ((unsigned long long)__popc(eqb[w0 + i]) << 32);
  unsigned long long total;
  const unsigned long long pre = block_scan_excl<unsigned long long>(cnt, sm.warp_sum64, &sm.total64, total);
  uint32_t gt_b = (uint32_t)(pre & 0xFFFFFFFFull), eq_b = (uint32_t)(pre >> 32);
  for (int i = 0; i < wpt && w0 + i < nw; ++i) {
    const uint32_t g = gtb[w0 + i], e = eqb[w0 + i];
    for (uint32_t mm = g | e; mm; mm &= mm - 1u) {
      const int b = __ffs(mm) - 1;
      const int q = (w0 + i) * 32 + b;
      if ((g >> b) & 1u) {
        const uint32_t o = gt_b + min(eq_b, take_eq);
        if (o < (uint32_t)k) out[o] = q;
        ++gt_b;
      } else {
        if (eq_b < take_eq && gt_b + eq_b < (uint32_t)k) out[gt_b + eq_b] = q;
        ++eq_b;
      }
    }
  }
}

int launch_topk_cand(const Shape& s, const uint32_t* cand_key, const int32_t* cand_pos,
                     const uint32_t* cand_cnt, long long ld, long long row_begin, long long rows,
                     int32_t* idx, DevCtx c, cudaStream_t st) {
  if (rows <= 0) return DSA_OK;
  const size_t marks = 2 * (size_t)((s.S_k + 31) / 32) * sizeof(uint32_t);
  if (marks > 48 * 1024 &&
      cudaFuncSetAttribute(topk_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)marks) !=
          cudaSuccess)
    return DSA_ERR_CUDA;
  topk_cand_kernel<<<(unsigned)rows, TK_THREADS, marks, st>>>(s, cand_key, cand_pos, cand_cnt, ld,
                                                               row_begin, idx, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

bool make_tmap_f32_lines(CUtensorMap* tm, const float* base, uint64_t rows, uint64_t ld,
                         uint64_t lines, uint32_t box_lines);

int launch_topk(const Shape& s, const float* scores, long long ld, long long row_begin,
                long long rows, int32_t* idx, DevCtx c, cudaStream_t st) {
  if (rows <= 0) return DSA_OK;
  const int max_n = s.S_k;
  if (max_n > 32768) {
    topk_stream_kernel<<<(int)rows, TK_THREADS, 0, st>>>(s, scores, ld, row_begin, idx, c);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  int dev = 0, sms = 0;  // the current device's SM count (queried per call: devices may differ)
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return DSA_ERR_CUDA;
  // The longest row of this launch sizes the block.  Rows of up to 4096 keys
  // take 256-thread blocks, four rows per SM (measured per 1824-row wave:
  // 45 us at n <= 3648).  Longer rows take one 1024-thread block per SM,
  // whose cost per row hardly depends on the row's length (the select's
  // barrier phases dominate): up to 16384 keys as two 512-thread groups with
  // a row each (16 keys per thread up to 8192, 32 up to 16384), so one row's
  // barrier phases overlap the other's work, beyond that one row over all
  // 1024 threads (32 keys each).  Measured per wave: one row over 1024
  // threads 67-69 us (8 keys per thread, 4K-8K keys) and 78-84 us (16 keys,
  // 8K-16K keys); 256-thread blocks with 32 keys 72-86 us at 4K-8K keys;
  // separate 512-thread blocks, two per SM, without the TMA stage 100-145 us
  // at 8K-16K keys.  The 1024-thread blocks stage each group's next row by TMA.
  long long n_rows_max = max_n;
  if (s.q_row_index == nullptr) {
    const long long b0 = row_begin / s.S_q, b1 = (row_begin + rows - 1) / s.S_q;
    const long long pmax = s.q_row_offset + (b0 == b1 ? (row_begin + rows - 1) % s.S_q : s.S_q - 1);
    n_rows_max = pmax + 1 < max_n ? pmax + 1 : max_n;
    if (n_rows_max < 1) n_rows_max = 1;
    // rows of one batch that cross 16384 keys: the rows up to 16384 keys go
    // to the two-group form in a launch of their own (when they fill at
    // least one round of it), the longer ones to the one-row form
    const long long n0 = s.q_row_offset + row_begin % s.S_q + 1;  // the first row's keys
    if (n_rows_max > 16384 && b0 == b1 && n0 <= 16384) {
      const long long lo = 16384 - n0 + 1;
      if (lo >= 2LL * sms && lo < rows) {
        const int rc = launch_topk(s, scores, ld, row_begin, lo, idx, c, st);
        if (rc != DSA_OK) return rc;
        return launch_topk(s, scores + lo * ld, ld, row_begin + lo, rows - lo, idx + lo * s.topk, c, st);
      }
    }
  }
  const int nt = n_rows_max <= 4096 ? 256 : 1024;
  const int groups = nt == TK_THREADS && n_rows_max <= 16384 ? 2 : 1;
  int kpt = groups == 2 && n_rows_max <= 8192 ? 16 : 32;
  if (nt == 256) kpt = n_rows_max <= 1024 ? 4 : n_rows_max <= 2048 ? 8 : 16;
  const long long per_sm = TK_THREADS / nt;                     // CTAs per SM
  const long long units = (rows + groups - 1) / groups;         // row groups
  const int g = (int)(units < per_sm * sms ? units : per_sm * sms);
  // TMA view of each row (1024-thread form): S_k / 32 lines of 32 floats (the
  // last S_k % 32 columns, if any, are read directly)
  CUtensorMap tm;
  memset(&tm, 0, sizeof(tm));
  int tma_elems = 0;
  if (nt == TK_THREADS && (reinterpret_cast<uintptr_t>(scores) & 15u) == 0 && ld % 4 == 0 &&
      max_n >= 32) {
    const uint32_t box_lines = 32 * kpt < 256 ? 32 * kpt : 256;
    if (!make_tmap_f32_lines(&tm, scores, (uint64_t)rows, (uint64_t)ld, (uint64_t)(max_n / 32),
                             box_lines))
      return DSA_ERR_CUDA;
    tma_elems = (max_n / 32) * 32;
  }
  const size_t stage = nt == TK_THREADS ? (size_t)(nt / groups) * kpt * 4 : 0;
  const size_t per_group = groups == 2 ? sizeof(TopkRegSmemT<TK_CAND / 2>) : sizeof(TopkRegSmemT<TK_CAND>);
  const size_t smem = 1024 + groups * (stage + per_group);
  auto run = [&](auto kernel) -> int {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return DSA_ERR_CUDA;
    kernel<<<g, nt, smem, st>>>(tm, s, scores, ld, row_begin, rows, idx, c, tma_elems);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  };
  if (nt == 256) {
    if (kpt == 4) return run(topk_reg_kernel<4, 256, 1>);
    if (kpt == 8) return run(topk_reg_kernel<8, 256, 1>);
    return run(topk_reg_kernel<16, 256, 1>);
  }
  if (groups == 2) {
    if (kpt == 16) return run(topk_reg_kernel<16, 1024, 2>);
    return run(topk_reg_kernel<32, 1024, 2>);
  }
  return run(topk_reg_kernel<32, 1024, 1>);
}

}  // namespace dsa
