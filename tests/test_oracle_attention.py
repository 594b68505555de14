"""Pins for the oracle's sparse attention forward (CPU only)."""
import numpy as np
import torch
import torch.nn.functional as F

from oracle import positions, sparse_attn_fwd, topk_select, indexer_scores


def test_hand_example(golden):
    g = golden("attention_hand.json")
    O, m, l = sparse_attn_fwd(np.array(g["q"]), np.array(g["kv"]), np.array(g["idx"]), g["scale"], g["d_v"])
    np.testing.assert_allclose(O, np.array(g["expected_O"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(m, np.array(g["expected_m"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, np.array(g["expected_l"]), rtol=0, atol=1e-15)


def _rand(B, S, H, d_qk, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, S, H, d_qk)), rng.standard_normal((B, S, d_qk))


def test_dense_limit_equals_causal_sdpa():
    # top-k >= causal length selects every visible key: dense causal softmax
    # attention (torch's SDPA in fp64, K = kv, V = kv[..., :d_v], all heads share them).
    B, S, H, d_qk, d_v = 2, 23, 3, 10, 6
    scale = 0.37
    q, kv = _rand(B, S, H, d_qk, 11)
    idx = np.full((B, S, S + 3), -1, dtype=np.int32)
    for t in range(S):
        idx[:, t, :t + 1] = np.arange(t + 1)
    O, m, l = sparse_attn_fwd(q, kv, idx, scale, d_v)
    qt = torch.from_numpy(q).transpose(1, 2)                      # [B,H,S,d]
    kt = torch.from_numpy(kv)[:, None].expand(B, H, S, d_qk)
    vt = kt[..., :d_v]
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale).transpose(1, 2)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-12, atol=1e-12)
    logits = scale * torch.einsum("bhsd,bhtd->bhst", qt, kt)
    logits = logits.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(m, logits.amax(-1).transpose(1, 2).numpy(), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(l, torch.exp(logits - logits.amax(-1, keepdim=True)).sum(-1)
                               .transpose(1, 2).numpy(), rtol=1e-12)


def test_single_key_returns_its_value_row():
    B, S, H, d_qk, d_v = 1, 9, 4, 7, 5
    q, kv = _rand(B, S, H, d_qk, 12)
    idx = np.full((B, S, 3), -1, dtype=np.int32)
    idx[0, :, 1] = np.arange(S)[::-1] % (np.arange(S) + 1)
    O, m, l = sparse_attn_fwd(q, kv, idx, 0.5, d_v)
    for t in range(S):
        s = idx[0, t, 1]
        np.testing.assert_allclose(O[0, t], np.broadcast_to(kv[0, s, :d_v], (H, d_v)), atol=1e-15)
        np.testing.assert_allclose(l[0, t], 1.0)
        np.testing.assert_allclose(m[0, t], 0.5 * q[0, t] @ kv[0, s], rtol=1e-14)


def test_softmax_rows_sum_to_one_and_order_invariance():
    B, S, H, d_qk, d_v, k = 1, 40, 4, 12, 8, 7
    q, kv = _rand(B, S, H, d_qk, 13)
    rng = np.random.default_rng(0)
    sc = rng.standard_normal((B, S, S)).astype(np.float32)
    pos = positions(B, S)
    idx = topk_select(sc, pos, k)
    scale = 0.3
    O, m, l = sparse_attn_fwd(q, kv, idx, scale, d_v)
    for t in range(S):
        sel = idx[0, t][idx[0, t] >= 0]
        s = scale * q[0, t] @ kv[0, sel].T
        np.testing.assert_allclose(np.exp(s - m[0, t][:, None]).sum(1) / l[0, t], 1.0, rtol=1e-13)
    # the order of the indices and extra padding do not matter
    idx2 = np.full((B, S, k + 5), -1, dtype=np.int32)
    for t in range(S):
        sel = idx[0, t][idx[0, t] >= 0][::-1]
        idx2[0, t, 2:2 + sel.size] = sel
    O2, m2, l2 = sparse_attn_fwd(q, kv, idx2, scale, d_v)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(m2, m, rtol=0, atol=0)
