"""CPU oracle for the DeepSeek Sparse Attention (DSA) hot path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The library never calls it and shares no
code with it: the CUDA path lives in ``sparse_attention_long_gb300/csrc`` and
nothing here is imported there or vice versa.

Plain, slow, per-query-row loops in float64 (numpy).  A matrix product, an
exponential or a stable sort from numpy is the only library help; there is no
blocking, fusion or reordering beyond the definitions.  Inputs are the exact
values of the bf16 / fp32 tensors the GPU path receives, widened to float64.

Sources (pages; titles abbreviated as below):

* [DSA-32K]  "CANN&TorchTitan: DeepSeek-V3.2 32k long-sequence pretraining on
  Ascend" -- section "DSA fused ops / SparseLightningIndexerGradKLLoss"
  (Lightning Indexer forward formula; Sparse Flash Attention forward formula;
  KL loss; dI; dW / dq~ / dK~ formulas) and section "SparseFlashAttentionGrad"
  (Gather, recompute softmax, dP, dS, dQ, dK, dV formulas).
* [HP-CP]    "CP context parallel guide" (HyperParallel context_parallel.md) --
  section "DSA CP" (operator boundaries, Shard(seq) / Replicate placements,
  BSND/TND layouts) and the ``load_balance`` parameter note (head-tail Q swap,
  mask built from K's length).
* [NPU-ops]  "CANN/torchtitan-npu fused-operator adaptation" -- section
  "DSA (DeepSeek Sparse Attention)": the indexer selects a few high-value
  tokens whose indices drive the sparse multi-query attention.

Readings taken where the pages are silent or garbled (each is listed in the
design notes as well):

* indexer scores are taken over every causal key s <= pos(t); the top-k form on
  the page is the loss-stage restriction.  No extra scale in the formula.
* causal: key s is visible to the query at global position p iff s <= p; the
  key length is the global length (the load_balance note).
* top-k order key: value descending, then index ascending; -0.0 == +0.0;
  output sorted by ascending index, padded with -1 when fewer than k keys
  are visible.  One index set per query token, shared by all heads.
* V is the first d_v columns of the shared kv row (MLA weight absorption).
* softmax_max / softmax_sum: natural exp over the scaled logits,
  m = max_i scale*q.k_i, l = sum_i exp(scale*q.k_i - m), valid selected keys.
* the KL target p sums the attention probabilities over heads, then
  L1-normalises along the selected keys; the indexer softmax runs over the
  same selected keys; the loss sums over query tokens; 0 log 0 = 0; p is a
  detached target.  ReLU'(0) = 0.
* FlashSoftmaxGrad(dY, O) is the row sum D = sum_e dY*O; dK and dV of the
  shared kv row are added into one dKV; dQ and dK both carry ``scale``.

Parity pins: every public function here is pinned by the CPU tests in
``tests/test_oracle_*.py`` (hand-derived closed forms in ``tests/golden/``,
library routines on special cases, finite differences, brute force).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    """torch tensor or array -> float64 numpy array (exact widening)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if x.dtype.is_floating_point:
            x = x.double()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.asarray(x, dtype=np.int64)


def positions(B: int, S_q: int, q_row_offset: int = 0, q_row_index=None) -> np.ndarray:
    """Global position of every local query row, [B, S_q] int64.

    [HP-CP] "DSA CP": the query side is Shard(seq) and the key side is
    Replicate(), so local row t of a shard sits at a global position; with
    head-tail balancing (load_balance) a rank owns two non-adjacent chunks, so
    the position is an explicit per-row list.  pos(t) = q_row_index[t] if given,
    else q_row_offset + t.
    """
    if q_row_index is not None:
        p = _i64(q_row_index).reshape(B, S_q)
        return p.copy()
    return np.broadcast_to(q_row_offset + np.arange(S_q, dtype=np.int64), (B, S_q)).copy()


def indexer_scores(q_I, k_I, w, pos) -> np.ndarray:
    """Lightning Indexer scores, [B, S_q, S_k] float64, -inf where s > pos(t).

    [DSA-32K] SparseLightningIndexerGradKLLoss, Lightning Indexer forward:
    I[t, s] = sum_j W[t, j] * ReLU(q~[t, j, :] . k~[s, :])  over the G index heads
    j of token t, one index key per position (MQA).  Evaluated for every causal
    key s <= pos(t) (reading: the top-k restriction on the page is the loss
    stage).  q_I [B,S_q,H_I,d_I], k_I [B,S_k,d_I], w [B,S_q,H_I].
    """
    q_I, k_I, w, pos = _f64(q_I), _f64(k_I), _f64(w), _i64(pos)
    B, S_q = q_I.shape[:2]
    S_k = k_I.shape[1]
    out = np.full((B, S_q, S_k), -np.inf)
    for b in range(B):
        for t in range(S_q):
            n = int(pos[b, t]) + 1
            S = q_I[b, t] @ k_I[b, :n].T              # [H_I, n]  index logits
            out[b, t, :n] = w[b, t] @ np.maximum(S, 0.0)
    return out


def topk_select(scores, pos, k: int) -> np.ndarray:
    """Per-query top-k indices, [B, S_q, k] int32.

    [DSA-32K] "Top-k positions of each token" feed the gather of K_topk;
    [NPU-ops] the indexer keeps a few high-value tokens.  Reading: among keys
    s <= pos(t), order by value descending then index ascending (-0.0 equals
    +0.0); keep the first min(k, pos(t)+1); emit them in ascending index order;
    pad with -1.  ``scores`` is compared in the dtype it is given in.
    """
    if hasattr(scores, "detach"):
        sc = scores.detach().to("cpu").numpy()
    else:
        sc = np.asarray(scores)
    pos = _i64(pos)
    B, S_q = sc.shape[:2]
    out = np.full((B, S_q, k), -1, dtype=np.int32)
    for b in range(B):
        for t in range(S_q):
            n = int(pos[b, t]) + 1
            row = sc[b, t, :n]
            order = np.argsort(-row, kind="stable")   # desc value, asc index on ties
            keep = np.sort(order[:min(k, n)])
            out[b, t, :keep.size] = keep
    return out


def _valid(idx_row):
    return idx_row[idx_row >= 0]


def sparse_attn_fwd(q, kv, idx, scale: float, d_v: int):
    """Sparse multi-query attention over the selected kv rows.

    [DSA-32K] Sparse Flash Attention forward: p[t,:] = Softmax(q[t,:] K_topk^T / sqrt(d))
    with K_topk the rows picked by token t's top-k indices; all heads of the
    token share them.  Output O = p V_topk with V = the first d_v columns of the
    shared kv row (weight-absorbed MLA).  Two-pass softmax per (t, h):
    m = max_i s_i, l = sum_i exp(s_i - m), s_i = scale * q[t,h] . kv[idx_i].

    q [B,S_q,H,d_qk], kv [B,S_k,d_qk], idx [B,S_q,k] (-1 = padding).
    Returns O [B,S_q,H,d_v], softmax_max [B,S_q,H], softmax_sum [B,S_q,H].
    """
    q, kv, idx = _f64(q), _f64(kv), _i64(idx)
    B, S_q, H, _ = q.shape
    O = np.zeros((B, S_q, H, d_v))
    m = np.full((B, S_q, H), -np.inf)
    l = np.zeros((B, S_q, H))
    for b in range(B):
        for t in range(S_q):
            sel = _valid(idx[b, t])
            if sel.size == 0:
                continue
            K = kv[b, sel]                              # [n, d_qk]
            s = scale * (q[b, t] @ K.T)                 # [H, n]
            mt = s.max(axis=1)
            e = np.exp(s - mt[:, None])
            lt = e.sum(axis=1)
            O[b, t] = (e / lt[:, None]) @ K[:, :d_v]
            m[b, t], l[b, t] = mt, lt
    return O, m, l


def sparse_attn_bwd(q, kv, idx, O, dO, m, l, scale: float, d_v: int):
    """Backward of the sparse attention.

    [DSA-32K] SparseFlashAttentionGrad: K_topk = Gather(K, idx); recompute
    P = Softmax(Q K_topk^T / sqrt(d)) (here from the saved m, l);
    dP = dY V^T; dS = P * (dP - FlashSoftmaxGrad(dY, O)) with
    FlashSoftmaxGrad = D = sum_e dY*O per (t, h); dQ = dS K_topk * scale;
    dK = ScatterAdd(dS^T Q * scale, idx); dV = P^T dY.  K and V alias the same
    kv row, so dK (all d_qk columns) and dV (first d_v columns) add into dKV.
    Returns dq [B,S_q,H,d_qk], dkv [B,S_k,d_qk].
    """
    q, kv, idx = _f64(q), _f64(kv), _i64(idx)
    O, dO, m, l = _f64(O), _f64(dO), _f64(m), _f64(l)
    B, S_q, H, d_qk = q.shape
    dq = np.zeros_like(q)
    dkv = np.zeros_like(kv)
    for b in range(B):
        for t in range(S_q):
            sel = _valid(idx[b, t])
            if sel.size == 0:
                continue
            K = kv[b, sel]
            V = K[:, :d_v]
            s = scale * (q[b, t] @ K.T)
            P = np.exp(s - m[b, t][:, None]) / l[b, t][:, None]   # [H, n]
            D = (dO[b, t] * O[b, t]).sum(axis=1)                  # [H]
            dP = dO[b, t] @ V.T                                   # [H, n]
            dS = P * (dP - D[:, None])
            dq[b, t] = scale * (dS @ K)
            dK = scale * (dS.T @ q[b, t])                         # [n, d_qk]
            dV = P.T @ dO[b, t]                                   # [n, d_v]
            np.add.at(dkv[b], sel, dK)
            dkv[b, sel, :d_v] += dV          # sel is unique within a row
    return dq, dkv


def indexer_kl_loss(q, kv, idx, m, l, scale: float, q_I, k_I, w):
    """Indexer KL loss and its gradients w.r.t. q_I, k_I, w.

    [DSA-32K] SparseLightningIndexerGradKLLoss:
      * target p[t,:]: attention probabilities of token t (recomputed from the
        saved softmax max/sum) summed over all heads, then L1-normalised along
        the context (the selected keys);
      * Loss = sum_t D_KL(p[t,:] || Softmax(I[t,:])), D_KL(a||b) = sum a log(a/b),
        with I[t,i] = sum_j W[t,j] ReLU(S[t,j,i]), S = q~ . k~_topk^T;
      * dI[t,:] = Softmax(I[t,:]) - p[t,:];
      * dW[t,:] = dI[t,:] ReLU(S[t,:,:])^T;  dS = dI * W * 1[S > 0];
        dq~[t] = dS K~_topk;  dK~_topk += dS^T q~[t] (accumulated per index).
    Returns (loss, dq_I [B,S_q,H_I,d_I], dk_I [B,S_k,d_I], dw [B,S_q,H_I]).
    """
    q, kv, idx = _f64(q), _f64(kv), _i64(idx)
    m, l = _f64(m), _f64(l)
    q_I, k_I, w = _f64(q_I), _f64(k_I), _f64(w)
    B, S_q = q.shape[:2]
    loss = 0.0
    dq_I = np.zeros_like(q_I)
    dk_I = np.zeros_like(k_I)
    dw = np.zeros_like(w)
    for b in range(B):
        for t in range(S_q):
            sel = _valid(idx[b, t])
            if sel.size == 0:
                continue
            s = scale * (q[b, t] @ kv[b, sel].T)                  # [H, n]
            P = np.exp(s - m[b, t][:, None]) / l[b, t][:, None]
            ph = P.sum(axis=0)                                     # sum over heads
            p = ph / ph.sum()                                      # L1 along context
            S = q_I[b, t] @ k_I[b, sel].T                         # [H_I, n]
            R = np.maximum(S, 0.0)
            I = w[b, t] @ R                                        # [n]
            z = I - I.max()
            logpi = z - np.log(np.exp(z).sum())
            pi = np.exp(logpi)
            nz = p > 0
            loss += float((p[nz] * (np.log(p[nz]) - logpi[nz])).sum())
            dI = pi - p
            dw[b, t] = R @ dI
            dS = (w[b, t][:, None] * dI[None, :]) * (S > 0)        # [H_I, n]
            dq_I[b, t] = dS @ k_I[b, sel]
            np.add.at(dk_I[b], sel, dS.T @ q_I[b, t])
    return loss, dq_I, dk_I, dw


def dsa_forward(q_I, k_I, w, q, kv, k: int, scale: float, d_v: int,
                q_row_offset: int = 0, q_row_index=None):
    """Whole forward: indexer scores -> top-k -> sparse attention.

    [NPU-ops] DSA section: the Lightning Indexer picks the indices used by the
    sparse multi-query attention; [HP-CP] DSA CP: a query shard attends the
    full (replicated) key side at its global positions.
    Returns (scores, idx, O, m, l).
    """
    B, S_q = q.shape[:2]
    pos = positions(B, S_q, q_row_offset, q_row_index)
    scores = indexer_scores(q_I, k_I, w, pos)
    idx = topk_select(scores, pos, k)
    O, m, l = sparse_attn_fwd(q, kv, idx, scale, d_v)
    return scores, idx, O, m, l
