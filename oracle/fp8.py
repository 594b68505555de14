"""CPU oracle for the FP8 (E4M3) Lightning Indexer -- TEST INFRASTRUCTURE.

Only the tests may import this module; the library never calls it and shares
no code with it.

The pages mention FP8 only for the MoE layers ([DSA-32K], "Why TorchTitan":
TorchAO FP8 / MxFP8) and give no DSA FP8 recipe, so this module states one
reading and computes it plainly:

* q_I and k_I are quantized per 128-element vector (one vector per query
  token and index head, one per key) to E4M3 -- the FP8 format with 1 sign
  bit, 4 exponent bits (bias 7) and 3 mantissa bits whose largest finite
  value is 448 and which has no infinities;
* the vector's scale is absmax / 448 in fp32 (an all-zero vector takes scale
  1), each element is x / scale in fp32, rounded to the nearest E4M3 value
  (ties to the even mantissa) and clamped to +-448;
* the score is the Lightning Indexer formula of [DSA-32K] ("DSA fused ops /
  SparseLightningIndexerGradKLLoss", Lightning Indexer forward) on the
  dequantized vectors: I[t,s] = sum_j w[t,j] ReLU(sq[t,j] sk[s] (q8[t,j] . k8[s]));
  w stays bf16.  Top-k and the attention are unchanged.

Everything below is float64 on the exact values (the fp32 steps of the
quantization are done in numpy float32, which rounds like the GPU).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6      # smallest normal binade: 2^-6
_MANT_BITS = 3


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value of each element (ties to even mantissa), clamped to
    +-448.  Input: exact float values (float32 or float64); output float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    # binade of each value; below the smallest normal binade the quantum is
    # that of the subnormals (2^-9)
    e = np.full(a.shape, _MIN_NORMAL_EXP, dtype=np.int64)
    e[nz] = np.maximum(np.floor(np.log2(a[nz])).astype(np.int64), _MIN_NORMAL_EXP)
    # guard the floor(log2) against rounding at exact powers of two
    e = np.where(nz & (np.ldexp(1.0, e) > a), e - 1, e)
    e = np.where(nz & (np.ldexp(1.0, e + 1) <= a), e + 1, e)
    e = np.maximum(e, _MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, e - _MANT_BITS)
    y = np.rint(a / quantum) * quantum        # a / quantum is exact; rint = half to even
    y = np.minimum(y, E4M3_MAX)
    out[nz] = y[nz]
    return np.copysign(out, x)


def quantize_rows(v):
    """Per-vector E4M3 quantization along the last axis (128 elements).
    Returns (codes as float64 values, scales as float64 of fp32 values)."""
    v32 = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v32), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    ratio = (v32 / scale[..., None]).astype(np.float32)   # fp32 division, round to nearest
    return e4m3_round(ratio), scale.astype(np.float64)


def indexer_scores_fp8(q_I, k_I, w, pos) -> np.ndarray:
    """FP8 Lightning Indexer scores over every causal key (the reading above).

    q_I [B,S_q,H_I,d_I], k_I [B,S_k,d_I], w [B,S_q,H_I] (bf16 values),
    pos [B,S_q] global positions.  Returns I [B,S_q,S_k] float64 with -inf at
    keys s > pos (not visible)."""
    def f64(x):
        if hasattr(x, "detach"):
            x = x.detach().to("cpu").float().numpy()
        return np.asarray(x, dtype=np.float64)
    qI, kI, w = f64(q_I), f64(k_I), f64(w)
    pos = np.asarray(pos)
    B, S_q, H_I, _ = qI.shape
    S_k = kI.shape[1]
    q8, sq = quantize_rows(qI)              # [B,S_q,H_I,d], [B,S_q,H_I]
    k8, sk = quantize_rows(kI)              # [B,S_k,d], [B,S_k]
    out = np.full((B, S_q, S_k), -np.inf)
    for b in range(B):
        for t in range(S_q):
            n = int(pos[b, t]) + 1
            if n <= 0:
                continue
            dots = q8[b, t] @ k8[b, :n].T                       # [H_I, n], exact products
            logits = sq[b, t][:, None] * sk[b, :n][None, :] * dots
            out[b, t, :n] = w[b, t] @ np.maximum(logits, 0.0)
    return out
