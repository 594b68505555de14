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

__device__ __forceinline__ void write_prefix_rows(int32_t* out, int n, int k) {
  for (int j = threadIdx.x; j < k; j += TK_THREADS) out[j] = j < n ? j : -1;
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

template <int VEC>
__global__ void __launch_bounds__(TK_THREADS, 1)
    topk_reg_kernel(Shape s, const float* __restrict__ scores, long long ld, long long row_begin,
                    int32_t* __restrict__ idx, DevCtx c) {
  __shared__ TopkSmem sm;
  const long long r_local = blockIdx.x;
  const long long row = row_begin + r_local;
  const int k = s.topk;
  int32_t* out = idx + r_local * (long long)k;
  const long long pos = row_pos(s, row);
  if (pos < 0 || pos >= s.S_k) {
    if (threadIdx.x == 0) set_status(c, DSA_ERR_INDEX);
    write_prefix_rows(out, 0, k);
    return;
  }
  const int n = (int)pos + 1;
  if (n <= k) {
    write_prefix_rows(out, n, k);
    return;
  }
  const float* src = scores + r_local * ld;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wbase = warp * 128 * VEC;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0);
  uint32_t key[VEC][4];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int e0 = wbase + j * 128 + lane * 4;
    if (vec_ok && e0 + 3 < n) {
      float4 v = __ldcs(reinterpret_cast<const float4*>(src + e0));
      key[j][0] = ordered_key(v.x);
      key[j][1] = ordered_key(v.y);
      key[j][2] = ordered_key(v.z);
      key[j][3] = ordered_key(v.w);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) key[j][q] = (e0 + q < n) ? ordered_key(__ldcs(src + e0 + q)) : 0u;
    }
  }
  auto for_each = [&](auto fn) {
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const int e0 = wbase + j * 128 + lane * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (e0 + q < n) fn(key[j][q]);
    }
  };
  int sh;
  uint32_t tp, take_eq;
  radix_select(sm, k, for_each, sh, tp, take_eq);

  // index-ordered compaction: packed (gt | eq << 16) counts
  uint32_t pre[VEC];
  uint32_t run = 0;
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int e0 = wbase + j * 128 + lane * 4;
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e0 + q < n) {
        const uint32_t kk = key[j][q] >> sh;
        cnt += (kk > tp) ? 1u : ((kk == tp) ? 0x10000u : 0u);
      }
    }
    uint32_t x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    pre[j] = run + x - cnt;
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  uint32_t total;
  const uint32_t wexcl = block_scan_excl<uint32_t>(lane == 0 ? run : 0u, sm.warp_sum, &sm.total, total);
  const uint32_t wbase_cnt = __shfl_sync(0xffffffffu, wexcl, 0);
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int e0 = wbase + j * 128 + lane * 4;
    uint32_t p = wbase_cnt + pre[j];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e0 + q < n) {
        const uint32_t kk = key[j][q] >> sh;
        const uint32_t gt_b = p & 0xFFFFu, eq_b = p >> 16;
        if (kk > tp) {
          const uint32_t o = gt_b + min(eq_b, take_eq);
          if (o < (uint32_t)k) out[o] = e0 + q;
          p += 1u;
        } else if (kk == tp) {
          if (eq_b < take_eq && gt_b + eq_b < (uint32_t)k) out[gt_b + eq_b] = e0 + q;
          p += 0x10000u;
        }
      }
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
    write_prefix_rows(out, 0, k);
    return;
  }
  const int n = (int)pos + 1;
  if (n <= k) {
    write_prefix_rows(out, n, k);
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

int launch_topk(const Shape& s, const float* scores, long long ld, long long row_begin,
                long long rows, int32_t* idx, DevCtx c, cudaStream_t st) {
  const int g = (int)rows;
  const int max_n = s.S_k;
  if (max_n <= 4096)
    topk_reg_kernel<1><<<g, TK_THREADS, 0, st>>>(s, scores, ld, row_begin, idx, c);
  else if (max_n <= 8192)
    topk_reg_kernel<2><<<g, TK_THREADS, 0, st>>>(s, scores, ld, row_begin, idx, c);
  else if (max_n <= 16384)
    topk_reg_kernel<4><<<g, TK_THREADS, 0, st>>>(s, scores, ld, row_begin, idx, c);
  else if (max_n <= 32768)
    topk_reg_kernel<8><<<g, TK_THREADS, 0, st>>>(s, scores, ld, row_begin, idx, c);
  else
    topk_stream_kernel<<<g, TK_THREADS, 0, st>>>(s, scores, ld, row_begin, idx, c);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
