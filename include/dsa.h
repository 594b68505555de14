/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention hot path.
 *
 * The path: Lightning Indexer scores -> per-query top-k -> sparse multi-query
 * attention (MLA weight-absorbed) over the selected kv rows, its backward, and
 * the indexer KL loss with its gradients.
 *
 * Sources (pages):
 *  [DSA-32K] "CANN&TorchTitan: DeepSeek-V3.2 32k long-sequence pretraining on
 *            Ascend", sections "DSA fused ops / SparseLightningIndexerGradKLLoss"
 *            and "SparseFlashAttentionGrad".
 *  [HP-CP]   "CP context parallel guide" (HyperParallel), section "DSA CP":
 *            the three DSA operator boundaries, Shard(seq) on the query side,
 *            Replicate() on the key side, layouts BSND / TND, mode "colossal".
 *  [NPU-ops] "CANN/torchtitan-npu fused-operator adaptation", section "DSA".
 *
 * Conventions shared by every call
 *  - Every tensor pointer is a DEVICE pointer owned by the caller (unless the
 *    argument says host).  The library never allocates, frees or synchronises
 *    the device (dsa_get_status excepted); all work is enqueued on `stream`
 *    (a cudaStream_t; NULL = legacy default stream).
 *  - Tensors are contiguous row-major in BSND order: [B, S, N(heads), D];
 *    TND is the same memory with B = 1.  "rows" are flattened (b, t) query
 *    rows r = b*S_q + t.
 *  - dtype DSA_BF16: q_I, k_I, w, q, kv, out, dout, dq, dq_I are bf16; index
 *    scores, softmax_max/sum, dkv, dk_I, dw, loss are fp32.  DSA_FP32: all
 *    floating tensors fp32 (exact-arithmetic path for small shapes).
 *  - The bf16 path is built for the DeepSeek-V3.2 shapes: H = 128,
 *    d_qk = 576 (512 latent + 64 rope), d_v = 512, H_I = 64, d_I = 128.
 *    and topk <= 2048 for the attention.  Other bf16 shapes return
 *    DSA_ERR_UNSUPPORTED.  The fp32 path takes any
 *    H <= 1024, d_qk <= 1024, d_v <= d_qk, H_I <= 256, d_I <= 512,
 *    topk <= 8192.
 *  - Query row t of a CP shard sits at global position
 *        pos(t) = q_row_index ? q_row_index[b*S_q + t] : q_row_offset + t
 *    and sees keys s <= pos(t) of the full S_k-long key side ([HP-CP] DSA CP:
 *    query Shard(seq), key Replicate(); the load_balance note: the mask uses
 *    K's length as the global length).  0 <= pos(t) < S_k is required.
 *  - Return value: DSA_OK or a negative DSA_ERR_* code.  Argument errors are
 *    found on the host before anything is enqueued and leave every output
 *    untouched.  Errors found on the device (a wait that ran out of time, an
 *    index out of range) set a device status word read by dsa_get_status.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dsa_stream_t; /* identical to cudaStream_t */

enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer      */
  DSA_ERR_UNSUPPORTED = -2, /* layout/mode/shape this library does not run     */
  DSA_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required      */
  DSA_ERR_CUDA = -4,        /* a CUDA launch or runtime call failed            */
  DSA_ERR_TIMEOUT = -5,     /* (device) a bounded wait ran out of time         */
  DSA_ERR_INDEX = -6        /* (device) a top-k index outside [-1, S_k)        */
};

enum { DSA_BSND = 0, DSA_TND = 1 };
enum { DSA_BF16 = 0, DSA_FP32 = 1 };
/* [HP-CP] DSA CP supports only mode "colossal" (all-gathered key side); mode
 * "ulysses" is an error there and is DSA_ERR_UNSUPPORTED here. */
enum { DSA_CP_COLOSSAL = 0, DSA_CP_ULYSSES = 1 };

/* dsa_params.flags: DSA_FLAG_CAUSAL_ONLY: dsa_indexer_scores(_fp8) writes
 * only the causal entries s <= pos(t) and leaves the rest of each score row
 * untouched.  DSA_FLAG_FP8_INDEXER: dsa_forward scores with the FP8 (E4M3)
 * indexer of dsa_indexer_scores_fp8 (DeepSeek indexer shapes, bf16).
 * DSA_FLAG_FUSED_TOPK: dsa_forward selects through dsa_indexer_topk (the
 * fused indexer + streaming top-k; bf16 DeepSeek indexer shapes, S_k < 65536,
 * not with DSA_FLAG_FP8_INDEXER); the indices are the same. */
enum { DSA_FLAG_CAUSAL_ONLY = 1, DSA_FLAG_FP8_INDEXER = 2, DSA_FLAG_FUSED_TOPK = 4 };

/* workspace queries (dsa_workspace_size `which`) */
enum {
  DSA_CALL_FORWARD = 0,
  DSA_CALL_ATTN_FWD = 1,
  DSA_CALL_ATTN_BWD = 2,
  DSA_CALL_KL_BWD = 3,
  DSA_CALL_BACKWARD = 4,
  DSA_CALL_INDEXER_TOPK = 5
};

typedef struct {
  int32_t layout;              /* DSA_BSND or DSA_TND (TND requires B == 1)            */
  int32_t dtype;               /* DSA_BF16 or DSA_FP32                                 */
  int32_t cp_mode;             /* DSA_CP_COLOSSAL (0)                                  */
  int32_t flags;               /* DSA_FLAG_* bits, 0 = defaults                        */
  int64_t B, S_q, S_k;         /* batch, local query rows, key length (global)         */
  int64_t H, d_qk, d_v;        /* attention heads, q/k width, value width (V = kv[:d_v]) */
  int64_t H_I, d_I;            /* indexer heads and width                              */
  int64_t topk;                /* k                                                    */
  float scale;                 /* softmax scale, e.g. 1/sqrt(192)                      */
  int32_t reserved1;
  int64_t q_row_offset;        /* global position of local row 0 (if no q_row_index)  */
  const int32_t *q_row_index;  /* optional device [B*S_q] global positions, or NULL   */
  int64_t wave_rows;           /* dsa_forward: rows per indexer/top-k wave; 0 = auto:
                                  as many as fit 256 MB of scores, rounded down to a
                                  multiple of 4 x the SM count; 1024 when not even
                                  that many fit.  bf16 backward calls: with
                                  0 < wave_rows < S_q, rows per pass (the passes
                                  run one after the other, each within one
                                  batch, and the workspace holds one pass); 0 or
                                  >= S_q: one pass over all rows */
} dsa_params;

/* Library version as 10000*major + 100*minor + patch. */
int dsa_version(void);

/* Bytes of device workspace a call needs (0 if none); `which` is a
 * DSA_CALL_* value.  Returns 0 for invalid params too (the call itself then
 * reports the error). */
size_t dsa_workspace_size(const dsa_params *p, int which);

/*
 * Lightning Indexer scores.  [DSA-32K] Lightning Indexer forward:
 *   I[t, s] = sum_j w[t, j] * ReLU(q_I[t, j, :] . k_I[s, :]),  s <= pos(t),
 * one index key per position shared by the H_I index heads (MQA).
 *   q_I    [B, S_q, H_I, d_I]   k_I [B, S_k, d_I]   w [B, S_q, H_I]
 *   scores [rows, S_k] fp32 for flattened rows [row_begin, row_begin+rows);
 *          entries s > pos(t) are written as -inf (left untouched with
 *          DSA_FLAG_CAUSAL_ONLY).
 * rows must not be 0; row_begin + rows <= B*S_q.
 */
int dsa_indexer_scores(const dsa_params *p, const void *q_I, const void *k_I, const void *w,
                       int64_t row_begin, int64_t rows, float *scores, dsa_stream_t stream);

/*
 * FP8 (E4M3) Lightning Indexer.  The pages give no DSA FP8 recipe (they name
 * FP8 / MxFP8 for the MoE layers only, [DSA-32K] "Why TorchTitan"); this is
 * one reading of it: q_I and k_I are quantized per 128-element vector to
 * E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite
 * value 448, no infinities) with scale = absmax / 448 in fp32 (1 for an
 * all-zero vector), each element x / scale rounded to nearest even and
 * clamped to +-448; the score is the Lightning Indexer formula on the
 * dequantized vectors:
 *   I[t, s] = sum_j w[t, j] * ReLU(sq[t, j] * sk[s] * (q8[t, j, :] . k8[s, :])).
 * DeepSeek indexer shapes only (H_I 64, d_I 128) and dtype DSA_BF16, else
 * DSA_ERR_UNSUPPORTED.
 *
 * dsa_indexer_quantize_fp8: q_I [B, S_q, H_I, 128] and k_I [B, S_k, 128]
 *   bf16 (16-byte aligned) -> q8 [B, S_q, H_I, 128] and k8 [B, S_k, 128] E4M3
 *   codes (16-byte aligned, caller-owned), q_scale [B, S_q, H_I] and
 *   k_scale [B, S_k] fp32.
 * dsa_indexer_scores_fp8: the scores of flattened rows [row_begin,
 *   row_begin + rows) from those buffers, w [B, S_q, H_I] bf16; output and
 *   flags as dsa_indexer_scores.  Dot products of E4M3 values are exact
 *   products accumulated in fp32.
 */
int dsa_indexer_quantize_fp8(const dsa_params *p, const void *q_I, const void *k_I, uint8_t *q8,
                             float *q_scale, uint8_t *k8, float *k_scale, dsa_stream_t stream);
int dsa_indexer_scores_fp8(const dsa_params *p, const uint8_t *q8, const float *q_scale,
                           const uint8_t *k8, const float *k_scale, const void *w, int64_t row_begin,
                           int64_t rows, float *scores, dsa_stream_t stream);

/*
 * Per-query top-k.  [DSA-32K] "Top-k positions of each token" select the kv
 * rows gathered by the sparse attention; [NPU-ops] the indexer keeps a few
 * high-value tokens.  For flattened rows [row_begin, row_begin+rows):
 * among s <= pos(t), the topk largest scores[r - row_begin, s]; order key
 * value descending, then index ascending (-0.0 == +0.0); written to
 * idx[(r - row_begin)*topk ...] in ascending index order; when
 * pos(t)+1 < topk the tail is -1.  Bit-exact (integer compares on an
 * order-preserving map of the fp32 bits).  NaN scores: unspecified order.
 *   scores [rows, S_k] fp32 (values at s > pos(t) are ignored; the buffer must
 *          hold all rows x S_k floats: whole 128-byte lines of a row may be read)
 *   idx [rows, topk] int32
 */
int dsa_topk(const dsa_params *p, const float *scores, int64_t row_begin, int64_t rows,
             int32_t *idx, dsa_stream_t stream);

/*
 * Fused Lightning Indexer + streaming top-k (the pages select "Top-k
 * positions of each token" inside the indexer stage: [DSA-32K] "DSA fused
 * ops", Lightning Indexer forward; [NPU-ops] "DSA").  For flattened rows
 * [row_begin, row_begin+rows) writes idx[(r - row_begin)*topk ...] exactly as
 * dsa_indexer_scores followed by dsa_topk would (same scores, same order key,
 * ascending indices, -1 tail), without a score matrix: while the indexer
 * streams a row's keys it keeps a running threshold no larger than the row's
 * k-th largest score seen so far and writes out only the keys at or above it
 * (key and position, 8 bytes each); an exact selection over those candidates
 * follows.  bf16 DeepSeek indexer shapes (H_I 64, d_I 128), S_k < 65536;
 * otherwise DSA_ERR_UNSUPPORTED.
 *   workspace: dsa_workspace_size(p, DSA_CALL_INDEXER_TOPK) bytes (candidate
 *   lists for one wave of wave_rows rows: 8 x wave_rows x S_k bytes plus
 *   counts), 16-byte aligned; the rows go through it in waves.
 */
int dsa_indexer_topk(const dsa_params *p, const void *q_I, const void *k_I, const void *w,
                     int64_t row_begin, int64_t rows, int32_t *idx, void *workspace,
                     dsa_stream_t stream);

/*
 * Sparse multi-query attention forward.  [DSA-32K] Sparse Flash Attention
 * forward: p[t] = Softmax(q[t] K_topk^T * scale), O = p V_topk; every head of a
 * token shares its index row; V = kv[..., :d_v] (weight absorption).
 *   q   [B, S_q, H, d_qk]   kv [B, S_k, d_qk]   idx [B, S_q, topk] int32
 *       (-1 = padding, skipped; other values must lie in [0, S_k): one outside
 *        is skipped and flags DSA_ERR_INDEX on the device)
 *   out [B, S_q, H, d_v]
 *   softmax_max / softmax_sum [B, S_q, H] fp32:
 *       m = max_i scale*q.k_i,  l = sum_i exp(scale*q.k_i - m) over valid i
 *       ([HP-CP] DSA indexer-loss boundary carries softmax_max/softmax_sum).
 *       A row with no valid index gives out = 0, m = -inf, l = 0.
 *   bf16 path: DeepSeek head shapes only (H 128, d_qk 576, d_v 512) with
 *       topk <= 2048, else DSA_ERR_UNSUPPORTED; q, kv and out 16-byte aligned,
 *       else DSA_ERR_INVALID_ARG.
 *   workspace: dsa_workspace_size(p, DSA_CALL_ATTN_FWD) bytes (may be NULL if 0).
 */
int dsa_sparse_attn_fwd(const dsa_params *p, const void *q, const void *kv, const int32_t *idx,
                        void *out, float *softmax_max, float *softmax_sum, void *workspace,
                        dsa_stream_t stream);

/*
 * Sparse attention backward.  [DSA-32K] SparseFlashAttentionGrad: gather
 * K_topk, recompute P from softmax_max/sum, dP = dO V^T,
 * dS = P * (dP - D) with D = sum_e dO*out (FlashSoftmaxGrad(dY, attention_in)),
 * dQ = scale * dS K_topk, dK = ScatterAdd(scale * dS^T Q), dV = P^T dO; K and
 * V alias the kv row, so both land in dkv.
 *   out, dout [B, S_q, H, d_v]   dq [B, S_q, H, d_qk] (written)
 *   dkv [B, S_k, d_qk] fp32: ACCUMULATED (+=) with atomics -- the caller
 *       zeroes it (or passes partial sums of other shards).
 *   workspace: dsa_workspace_size(p, DSA_CALL_ATTN_BWD) bytes (the fp32 path
 *       accumulates dkv in fp64 there first; NULL allowed when the size is 0).
 *   bf16 path: DeepSeek head shapes only (H 128, d_qk 576, d_v 512) with
 *       topk <= 2048 and topk % 8 == 0, else DSA_ERR_UNSUPPORTED; q, kv, out,
 *       dout, dq, dkv and the workspace 16-byte aligned.  The workspace holds
 *       P and scale*dS for every (row, head, slot) of one pass as bf16 hi/lo
 *       pairs plus D, i.e. 1024 * rows * topk + 512 * rows + 256 bytes with
 *       rows = all B * S_q rows (34 GB at 16384 rows, topk = 2048) or, with
 *       0 < wave_rows < S_q, rows = wave_rows (2.1 GB at 1024); it must stay
 *       untouched until the call's kernels have finished on `stream`.
 */
int dsa_sparse_attn_bwd(const dsa_params *p, const void *q, const void *kv, const int32_t *idx,
                        const void *out, const void *dout, const float *softmax_max,
                        const float *softmax_sum, void *dq, float *dkv, void *workspace,
                        dsa_stream_t stream);

/*
 * Indexer KL loss and its gradients.  [DSA-32K] SparseLightningIndexerGradKLLoss:
 * p[t] = attention probabilities (recomputed from softmax_max/sum) summed over
 * heads, L1-normalised over the selected keys; pi[t] = Softmax(I[t, idx]) over
 * the same keys; Loss = sum_t KL(p[t] || pi[t]); dI = pi - p;
 * dw = dI ReLU(S)^T; dq_I = dS k_I[idx]; dk_I[idx] += dS^T q_I with
 * dS = dI * w * 1[S > 0], S = q_I . k_I[idx]^T.  p is a detached target.
 *   loss  1 fp32, ACCUMULATED (+= this call's rows); caller zeroes.
 *   dq_I [B, S_q, H_I, d_I] written;  dw [B, S_q, H_I] fp32 written;
 *   dk_I [B, S_k, d_I] fp32 ACCUMULATED with atomics; caller zeroes.
 *   workspace: dsa_workspace_size(p, DSA_CALL_KL_BWD) bytes (fp32 path: fp64
 *       accumulation of dk_I; NULL allowed when the size is 0).
 *   bf16 path: the attention shapes of dsa_sparse_attn_bwd plus H_I 64,
 *       d_I 128, else DSA_ERR_UNSUPPORTED; q, kv, k_I, dk_I and the workspace
 *       16-byte aligned, dq_I 4-byte aligned, topk <= 2048.  The workspace
 *       holds the head-summed attention probabilities, fp32:
 *       4 * rows * topk + 256 bytes (rows: one pass, as for
 *       dsa_sparse_attn_bwd).
 */
int dsa_indexer_kl_loss_bwd(const dsa_params *p, const void *q, const void *kv, const void *q_I,
                            const void *k_I, const void *w, const int32_t *idx,
                            const float *softmax_max, const float *softmax_sum, float *loss,
                            void *dq_I, float *dk_I, float *dw, void *workspace,
                            dsa_stream_t stream);

/*
 * Whole backward of one training step: dsa_sparse_attn_bwd and
 * dsa_indexer_kl_loss_bwd in one call, with the results of calling the two
 * one after the other.  [DSA-32K] SparseFlashAttentionGrad recomputes the
 * attention probabilities P and SparseLightningIndexerGradKLLoss needs their
 * head sum as its target; here the attention pass writes that sum while it has
 * P at hand, so the KL pass does not recompute the attention logits.
 *   Arguments, layouts, accumulation (dkv, loss, dk_I are ACCUMULATED; dq,
 *   dq_I, dw written) and alignment as in the two calls above.
 *   workspace: dsa_workspace_size(p, DSA_CALL_BACKWARD) bytes (bf16 path:
 *       the attention backward's workspace followed by the [rows][topk] fp32
 *       target; fp32 path: the larger of the two calls' workspaces, used by
 *       each in turn).
 */
int dsa_backward(const dsa_params *p, const void *q, const void *kv, const int32_t *idx,
                 const void *out, const void *dout, const float *softmax_max,
                 const float *softmax_sum, const void *q_I, const void *k_I, const void *w,
                 void *dq, float *dkv, float *loss, void *dq_I, float *dk_I, float *dw,
                 void *workspace, dsa_stream_t stream);

/*
 * Whole forward: indexer scores -> top-k -> sparse attention, the S x S score
 * matrix streamed through a workspace ring of wave_rows x S_k fp32 (never
 * materialised whole).  Outputs as in the calls above; idx_out [B, S_q, topk].
 * With DSA_FLAG_FP8_INDEXER the scores come from the FP8 indexer (q_I and
 * k_I quantized once per call into the workspace after the ring).
 *   workspace: dsa_workspace_size(p, DSA_CALL_FORWARD) bytes.
 */
int dsa_forward(const dsa_params *p, const void *q_I, const void *k_I, const void *w,
                const void *q, const void *kv, int32_t *idx_out, void *out, float *softmax_max,
                float *softmax_sum, void *workspace, dsa_stream_t stream);
/* (dsa_forward with DSA_FLAG_FUSED_TOPK: the indexer and top-k of each wave
 * are dsa_indexer_topk's, and the workspace holds its candidate lists.) */

/*
 * Whole forward with no workspace argument (this library's own addition; the
 * pages have no counterpart).  For callers that cannot allocate device memory
 * -- plug-in or custom-operator hosts that pass only input and output
 * buffers, or latency-critical loops that must not call cudaMalloc or an
 * allocator -- the score ring lives in a 32 MiB device array inside the
 * library, held on every GPU that loads the library until the process exits.
 * Arguments and outputs as dsa_forward; the waves hold as many rows as fit the
 * ring (a multiple of 4).  The ring's address is looked up by the first call
 * made on each device (make that call before any stream capture) and again
 * only if the device's CUDA context changed since.  All calls share the ring:
 * calls that overlap on the GPU race on it.
 * Returns DSA_ERR_UNSUPPORTED when S_k > 2,097,152 (4 score rows would not
 * fit the ring) or with DSA_FLAG_FP8_INDEXER or DSA_FLAG_FUSED_TOPK; never
 * allocates or frees device memory.
 */
int dsa_forward_static_ws(const dsa_params *p, const void *q_I, const void *k_I, const void *w,
                          const void *q, const void *kv, int32_t *idx_out, void *out,
                          float *softmax_max, float *softmax_sum, dsa_stream_t stream);

/*
 * Device status.  Synchronises `stream`, then writes the device status word
 * of the current device to *device_status (DSA_OK, DSA_ERR_TIMEOUT or
 * DSA_ERR_INDEX) and clears it.  Returns DSA_ERR_CUDA if the stream reported
 * a CUDA error, else DSA_OK.
 * There is ONE status word per device, shared by every stream and host thread
 * that uses the library on it: the first device error since the last read
 * wins, whatever stream raised it.  Only `stream` is synchronised, so an error
 * raised by a kernel still running on another stream may be reported by a
 * later call, and this call clears errors of other streams too.  Callers
 * that run several streams read the status after synchronising all of them.
 */
int dsa_get_status(dsa_stream_t stream, int *device_status);

/*
 * Upper bound, in nanoseconds, on every spin-wait inside the kernels (an
 * mbarrier or a cluster peer); a wait that runs out sets DSA_ERR_TIMEOUT in
 * the status word and the kernel winds down and returns.  Default 2e9 (2 s).
 * Applies to launches enqueued after the call on the current device.
 */
int dsa_set_wait_budget_ns(uint64_t budget_ns);

/*
 * Self-test of the bounded wait: enqueues one tiny kernel that waits on an
 * mbarrier nothing will complete, with the given budget; the wait gives up,
 * records DSA_ERR_TIMEOUT in the status word and the kernel returns normally.
 */
int dsa_selftest_wait_timeout(uint64_t budget_ns, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_GB300_H */
