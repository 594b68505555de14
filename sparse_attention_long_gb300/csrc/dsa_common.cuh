// Device-side building blocks shared by the sm_103a kernels: bounded mbarrier
// waits, TMA (tile and gather4) copies, tcgen05 MMA / TMEM access, shared
// memory matrix descriptors, and the problem description passed to kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// ---------------------------------------------------------------------------
// problem description handed to every kernel (plain values, device pointers)
// ---------------------------------------------------------------------------
struct Shape {
  int B, S_q, S_k, H, d_qk, d_v, H_I, d_I, topk;
  float scale;
  long long q_row_offset;
  const int32_t* q_row_index;  // device [B*S_q] or nullptr
};

struct DevCtx {
  int* status;                 // device status word (first error wins)
  unsigned long long budget;   // ns per bounded wait
};

__device__ __forceinline__ long long row_pos(const Shape& s, long long row) {
  // global position of flattened query row `row` = b*S_q + t
  return s.q_row_index ? (long long)s.q_row_index[row] : s.q_row_offset + (row % s.S_q);
}

__device__ __forceinline__ void set_status(const DevCtx& c, int code) {
  atomicCAS(c.status, 0, code);
}

// ---------------------------------------------------------------------------
// numeric helpers
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// shared memory / mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Remote arrive that orders no earlier memory operation: the caller must make
// sure by other means that what it releases is no longer being read.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// acquire at cluster scope: for barriers completed by the peer CTA's arrives
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true once the phase with `parity` completed; false if the
// CTA-wide abort flag is raised or the time budget ran out (then the status
// word gets DSA_ERR_TIMEOUT and the abort flag is raised).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const DevCtx& c,
                                          volatile int* abort_flag) {
  if (CLUSTER ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (CLUSTER ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > c.budget) {
        set_status(c, DSA_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Same, for waits every lane of a warp performs: the outcome is made
// warp-uniform so the warp never splits ahead of a .sync.aligned instruction.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const DevCtx& c,
                                               volatile int* abort_flag) {
  const bool ok = mbar_wait<CLUSTER>(bar, parity, c, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t mapa_shared(uint32_t local_addr, uint32_t cta_rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(cta_rank));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, uint32_t a, uint32_t b,
                                            uint32_t c, uint32_t d, uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(cluster_addr),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// cp.async gathers (16-byte global -> shared copies completing on an mbarrier)
// ---------------------------------------------------------------------------
// 16-byte global -> shared copy that bypasses registers (L2 only)
__device__ __forceinline__ void cp_async16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// arrive on `bar` once every cp.async this thread issued before has landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// shared -> global tile store (bulk-group completion); the caller fences the
// generic-proxy writes of the tile (fence.proxy.async) before issuing it
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tm),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// every committed bulk store of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed bulk store of this thread has completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive once on `bar` when every tcgen05 op issued so far by this thread is done
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// tcgen05.ld writes its destination registers asynchronously: they hold the
// data only after tcgen05.wait::ld.  The compiler sees them as defined by the
// load statement, so plain arithmetic on them could be scheduled before the
// wait.  The waits below therefore take the destination arrays as in/out
// operands: every use is data-dependent on the wait.
#define DSA_RW8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                   "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : DSA_RW8(0), DSA_RW8(8), DSA_RW8(16), DSA_RW8(24)
               :
               : "memory");
}
// after a tmem_ld_wait: ties one more destination array to that wait
__device__ __forceinline__ void tmem_ld_also(uint32_t (&r)[32]) {
  asm volatile("" : DSA_RW8(0), DSA_RW8(8), DSA_RW8(16), DSA_RW8(24) : : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#define DSA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define DSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// lane = thread's TMEM lane, 32 consecutive 32-bit columns starting at taddr
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : DSA_R8(0), DSA_R8(8), DSA_R8(16), DSA_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      DSA_W8(0), DSA_W8(8), DSA_W8(16), DSA_W8(24)
      : "memory");
}

// 16 / 8 consecutive columns (same lane mapping as tmem_ld32); the caller
// ties the destinations to a following tcgen05.wait::ld (tmem_ld_also16/8)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : DSA_R8(0), DSA_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : DSA_R8(0)
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : DSA_RW8(0), DSA_RW8(8) : : "memory");
}
__device__ __forceinline__ void tmem_ld_also16(uint32_t (&r)[16]) {
  asm volatile("" : DSA_RW8(0), DSA_RW8(8) : : "memory");
}
__device__ __forceinline__ void tmem_ld_also8(uint32_t (&r)[8]) {
  asm volatile("" : DSA_RW8(0) : : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      DSA_W8(0), DSA_W8(8)
      : "memory");
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// Scatter-add of a warp's 32 rows x 32 fp32 columns: lane i holds row i's 32
// values (as a 32x32b TMEM load leaves them) and the address they add into
// (row_dst, nullptr to skip the row).  The block is transposed through a 4 KB
// warp-private shared scratch (16-byte chunks XOR-swizzled by row, so both
// the row-wise stores and the column-wise loads are conflict-free), so each
// reduction instruction covers four rows' whole 128-byte segments: L2 takes
// full-line vector reductions at about twice the rate of 32 rows' 16-byte
// pieces.  The caller owns the scratch for the duration of the call.
__device__ __forceinline__ void warp_scatter_add_32x32(uint32_t scratch, const uint32_t (&v)[32],
                                                       float* row_dst) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(scratch + lane * 128 + ((j ^ (lane & 7)) << 4)),
                 "r"(v[4 * j]), "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                 : "memory");
  __syncwarp();
  const int ch = lane & 7;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int r = 4 * p + (lane >> 3);
    float* d = reinterpret_cast<float*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(row_dst), r));
    uint32_t x0, x1, x2, x3;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                 : "r"(scratch + r * 128 + ((ch ^ (r & 7)) << 4))
                 : "memory");
    if (d != nullptr)
      red_add_v4(d + 4 * ch, __uint_as_float(x0), __uint_as_float(x1), __uint_as_float(x2),
                 __uint_as_float(x3));
  }
  __syncwarp();
}

// (w0, w1) * (x0, x1) + acc as one packed fp32x2 FMA (each lane rounds like
// fmaf); acc holds two floats, the first in the low half
__device__ __forceinline__ uint64_t ffma2(float w0, float w1, float x0, float x1, uint64_t acc) {
  uint64_t w, x, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(w) : "f"(w0), "f"(w1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(w), "l"(x), "l"(acc));
  return d;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Half of the Lightning Indexer head reduction: heads h0 .. h0+31 (x in v,
// weights w[0..31]) added to the four running sums (heads j mod 4).
__device__ __forceinline__ void relu_acc32(const uint32_t (&v)[32], const float* w, uint64_t& a01,
                                           uint64_t& a23) {
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    const float4 wa = *reinterpret_cast<const float4*>(w + h);
    a01 = ffma2(wa.x, wa.y, fmaxf(__uint_as_float(v[h]), 0.f), fmaxf(__uint_as_float(v[h + 1]), 0.f), a01);
    a23 = ffma2(wa.z, wa.w, fmaxf(__uint_as_float(v[h + 2]), 0.f), fmaxf(__uint_as_float(v[h + 3]), 0.f), a23);
  }
}
__device__ __forceinline__ float relu_sum_finish(uint64_t a01, uint64_t a23) {
  float a0, a1, a2, a3;
  unpack2(a01, a0, a1);
  unpack2(a23, a2, a3);
  return (a0 + a1) + (a2 + a3);
}

// Lightning Indexer head reduction, sum_j w[j] * max(x_j, 0) over 64 heads,
// for the indexer epilogue's two tokens of one key block (lane = key): token
// 0's score from TMEM columns tb .. tb+63 (weights w0), token 1's from
// tb+64 .. tb+127 (w1).  Four running sums (heads j mod 4), advanced two at
// a time by packed FMAs, then (s0 + s1) + (s2 + s3).  The four 32-column
// pieces go through the caller's two register buffers A and B, so the next
// piece's TMEM load is in flight while the current piece is reduced; the
// first call returns token 0's score with token 1's first piece still
// loading (so its store overlaps that load), the second call token 1's.
__device__ __forceinline__ float relu_pair_first(uint32_t tb, const float* w0, uint32_t (&A)[32],
                                                 uint32_t (&B)[32]) {
  uint64_t a01 = 0, a23 = 0;
  tmem_ld32(tb, A);
  tmem_ld_wait(A);
  tmem_ld32(tb + 32, B);
  relu_acc32(A, w0, a01, a23);
  tmem_ld_wait(B);
  tmem_ld32(tb + 64, A);
  relu_acc32(B, w0 + 32, a01, a23);
  return relu_sum_finish(a01, a23);
}
__device__ __forceinline__ float relu_pair_second(uint32_t tb, const float* w1, uint32_t (&A)[32],
                                                  uint32_t (&B)[32]) {
  uint64_t a01 = 0, a23 = 0;
  tmem_ld_wait(A);
  tmem_ld32(tb + 96, B);
  relu_acc32(A, w1, a01, a23);
  tmem_ld_wait(B);
  relu_acc32(B, w1 + 32, a01, a23);
  return relu_sum_finish(a01, a23);
}

// Shared-memory matrix descriptor (tcgen05): start, leading / stride byte
// offsets, fixed version 1, swizzle layout (0 none, 2 = 128B, 4 = 64B, 6 = 32B).
constexpr uint32_t kSw128 = 2, kSw64 = 4;
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)layout << 61;
  return d;
}
// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// order-preserving map of fp32 bits to uint32 (-0.0 first folded onto +0.0)
__device__ __forceinline__ uint32_t ordered_key(float x) {
  // x + 0 turns -0 into +0 (IEEE round-to-nearest) and leaves every other
  // value unchanged; then negative values get all bits flipped, others the sign
  const uint32_t u = __float_as_uint(x + 0.0f);
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

}  // namespace dsa
