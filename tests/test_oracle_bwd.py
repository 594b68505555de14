"""Pins for the oracle's backward pieces (CPU only)."""
import numpy as np
import torch
import torch.nn.functional as F

from oracle import indexer_kl_loss, positions, sparse_attn_bwd, sparse_attn_fwd, topk_select


def test_attn_bwd_dense_limit_matches_autograd():
    B, S, H, d_qk, d_v, scale = 1, 17, 3, 10, 6, 0.31
    rng = np.random.default_rng(21)
    q = rng.standard_normal((B, S, H, d_qk))
    kv = rng.standard_normal((B, S, d_qk))
    dO = rng.standard_normal((B, S, H, d_v))
    idx = np.full((B, S, S), -1, dtype=np.int32)
    for t in range(S):
        idx[:, t, :t + 1] = np.arange(t + 1)
    O, m, l = sparse_attn_fwd(q, kv, idx, scale, d_v)
    dq, dkv = sparse_attn_bwd(q, kv, idx, O, dO, m, l, scale, d_v)
    qt = torch.from_numpy(q).requires_grad_(True)
    kvt = torch.from_numpy(kv).requires_grad_(True)
    k_ = kvt[:, None].expand(B, H, S, d_qk)
    out = F.scaled_dot_product_attention(qt.transpose(1, 2), k_, k_[..., :d_v], is_causal=True, scale=scale)
    out.transpose(1, 2).backward(torch.from_numpy(dO))
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dkv, kvt.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_attn_bwd_finite_differences_sparse():
    B, S, H, d_qk, d_v, k, scale = 1, 12, 2, 5, 3, 4, 0.45
    rng = np.random.default_rng(22)
    q = rng.standard_normal((B, S, H, d_qk))
    kv = rng.standard_normal((B, S, d_qk))
    dO = rng.standard_normal((B, S, H, d_v))
    idx = topk_select(rng.standard_normal((B, S, S)).astype(np.float32), positions(B, S), k)

    def f(q_, kv_):
        return float((sparse_attn_fwd(q_, kv_, idx, scale, d_v)[0] * dO).sum())

    O, m, l = sparse_attn_fwd(q, kv, idx, scale, d_v)
    dq, dkv = sparse_attn_bwd(q, kv, idx, O, dO, m, l, scale, d_v)
    eps = 1e-6
    for (arr, grad) in ((q, dq), (kv, dkv)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = arr[i]
            arr[i] = old + eps
            fp = f(q, kv)
            arr[i] = old - eps
            fm = f(q, kv)
            arr[i] = old
            assert abs((fp - fm) / (2 * eps) - grad[i]) < 1e-7, i


def test_kl_hand_example(golden):
    g = golden("kl_loss_hand.json")
    a = lambda n: np.array(g[n])
    loss, dq_I, dk_I, dw = indexer_kl_loss(a("q"), a("kv"), a("idx"), a("m"), a("l"), g["scale"],
                                           a("q_I"), a("k_I"), a("w"))
    assert abs(loss - g["expected_loss"]) < 1e-14
    np.testing.assert_allclose(dw, a("expected_dw"), atol=1e-15)
    np.testing.assert_allclose(dq_I, a("expected_dq_I"), atol=1e-15)
    np.testing.assert_allclose(dk_I, a("expected_dk_I"), atol=1e-15)


def test_kl_hand_example_two_heads(golden):
    # two heads with different softmax sums l: the target is the head sum of
    # each head's normalised probabilities (p = [3/8, 5/8] by hand)
    g = golden("kl_loss_hand_2heads.json")
    a = lambda n: np.array(g[n])
    loss, dq_I, dk_I, dw = indexer_kl_loss(a("q"), a("kv"), a("idx"), a("m"), a("l"), g["scale"],
                                           a("q_I"), a("k_I"), a("w"))
    assert abs(loss - g["expected_loss"]) < 1e-14
    np.testing.assert_allclose(dw, a("expected_dw"), atol=1e-15)
    np.testing.assert_allclose(dq_I, a("expected_dq_I"), atol=1e-15)
    np.testing.assert_allclose(dk_I, a("expected_dk_I"), atol=1e-15)
    # the same m, l with the second head's sum doubled must change the loss
    # (the target reads each head's own l)
    l2 = a("l").copy()
    l2[..., 1] *= 2.0
    assert abs(indexer_kl_loss(a("q"), a("kv"), a("idx"), a("m"), l2, g["scale"], a("q_I"), a("k_I"),
                               a("w"))[0] - g["expected_loss"]) > 1e-3


def _kl_case(seed, S=14, H=3, d_qk=6, H_I=2, d_I=4, k=5, scale=0.5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, S, H, d_qk))
    kv = rng.standard_normal((1, S, d_qk))
    qI = rng.standard_normal((1, S, H_I, d_I))
    kI = rng.standard_normal((1, S, d_I))
    w = rng.standard_normal((1, S, H_I))
    idx = topk_select(rng.standard_normal((1, S, S)).astype(np.float32), positions(1, S), k)
    _, m, l = sparse_attn_fwd(q, kv, idx, scale, 1)
    return q, kv, idx, m, l, scale, qI, kI, w


def test_kl_nonnegative_and_zero_when_distributions_match():
    for seed in range(5):
        assert indexer_kl_loss(*_kl_case(seed))[0] >= 0.0
    # one head, index query = scale*q and index key = kv with all logits > 0:
    # then I = the attention logits, Softmax(I) = p and the loss vanishes.
    rng = np.random.default_rng(9)
    S, d, scale = 8, 5, 0.7
    q = np.abs(rng.standard_normal((1, S, 1, d))) + 0.1
    kv = np.abs(rng.standard_normal((1, S, d))) + 0.1
    idx = np.tile(np.arange(S, dtype=np.int32), (1, S, 1))
    idx[0][np.triu(np.ones((S, S), dtype=bool), 1)] = -1
    _, m, l = sparse_attn_fwd(q, kv, idx, scale, 1)
    loss, dqI, dkI, dw = indexer_kl_loss(q, kv, idx, m, l, scale, scale * q, kv, np.ones((1, S, 1)))
    assert abs(loss) < 1e-13
    assert np.abs(dqI).max() < 1e-13 and np.abs(dkI).max() < 1e-13 and np.abs(dw).max() < 1e-13


def test_kl_finite_differences():
    q, kv, idx, m, l, scale, qI, kI, w = _kl_case(31)
    loss, dqI, dkI, dw = indexer_kl_loss(q, kv, idx, m, l, scale, qI, kI, w)
    eps = 1e-6
    f = lambda: indexer_kl_loss(q, kv, idx, m, l, scale, qI, kI, w)[0]
    S_all = np.einsum("btjd,bsd->btjs", qI, kI)
    assert np.abs(S_all).min() > 1e-4          # away from ReLU kinks
    for arr, grad in ((qI, dqI), (kI, dkI), (w, dw)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = arr[i]
            arr[i] = old + eps
            fp = f()
            arr[i] = old - eps
            fm = f()
            arr[i] = old
            assert abs((fp - fm) / (2 * eps) - grad[i]) < 1e-7, i


def test_kl_logit_gradient_sums_to_zero():
    # dI = Softmax(I) - p sums to 0 over a token's selected keys (both are
    # distributions).  Seen through dw: an index head whose score is the same
    # positive constant c for every key adds c to all logits, so its weight's
    # gradient is c * sum_i dI_i = 0, whatever the other heads do.
    q, kv, idx, m, l, scale, qI, kI, w = _kl_case(17)
    qI = qI.copy()
    kI = kI.copy()
    qI[..., 0, :] = 0.0
    qI[..., 0, 0] = 1.0                      # head 0: q_I = e_0 for every token
    kI[..., 0] = 0.75                        # k_I[s, 0] = 0.75 for every key
    _, _, _, dw = indexer_kl_loss(q, kv, idx, m, l, scale, qI, kI, w)
    assert np.abs(dw[..., 0]).max() < 1e-14
    assert np.abs(dw[..., 1:]).max() > 1e-6  # the other heads do get gradient
