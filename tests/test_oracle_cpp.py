"""Pins for the C++ oracle (oracle/dsa_ref.cpp, CPU only).

Two independent implementations of the same definitions -- the numpy oracle
and the C++ oracle -- must agree to rounding (~1e-12), and the C++ oracle is
held to the same pins as the numpy one: the hand-worked fixtures, the dense
limit against torch's SDPA, finite differences of the gradients, exact top-k
on ties and signed zeros, and results independent of the thread count."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import cpp


@pytest.fixture(scope="module", autouse=True)
def built():
    cpp.build()


def _case(seed, B=1, S=40, H=3, d_qk=12, d_v=8, H_I=4, d_I=6, k=9):
    rng = np.random.default_rng(seed)
    return dict(q_I=rng.standard_normal((B, S, H_I, d_I)), k_I=rng.standard_normal((B, S, d_I)),
                w=rng.standard_normal((B, S, H_I)), q=rng.standard_normal((B, S, H, d_qk)),
                kv=rng.standard_normal((B, S, d_qk)), dO=rng.standard_normal((B, S, H, d_v)),
                k=k, d_v=d_v, scale=0.41)


@pytest.mark.parametrize("seed,threads", [(0, 1), (1, 4), (2, 16)])
def test_forward_agrees_with_numpy_oracle(seed, threads):
    x = _case(seed, B=2)
    r_np = oracle.dsa_forward(x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], x["k"], x["scale"], x["d_v"])
    r_cc = cpp.dsa_forward(x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], x["k"], x["scale"], x["d_v"],
                           threads=threads)
    sc, idx, O, m, l = r_np
    fin = np.isfinite(sc)
    assert np.array_equal(fin, np.isfinite(r_cc[0]))
    np.testing.assert_allclose(r_cc[0][fin], sc[fin], rtol=1e-12, atol=1e-12)
    assert np.array_equal(r_cc[1], idx)
    np.testing.assert_allclose(r_cc[2], O, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r_cc[3], m, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r_cc[4], l, rtol=1e-12, atol=1e-12)


def test_cp_rows_agree_with_numpy_oracle():
    x = _case(3, S=48)
    rows = np.array([0, 1, 2, 45, 46, 47], dtype=np.int64)
    sel = lambda a: a[:, rows]
    r_np = oracle.dsa_forward(sel(x["q_I"]), x["k_I"], sel(x["w"]), sel(x["q"]), x["kv"], x["k"],
                              x["scale"], x["d_v"], q_row_index=rows)
    r_cc = cpp.dsa_forward(sel(x["q_I"]), x["k_I"], sel(x["w"]), sel(x["q"]), x["kv"], x["k"],
                           x["scale"], x["d_v"], q_row_index=rows, threads=3)
    assert np.array_equal(r_cc[1], r_np[1])
    np.testing.assert_allclose(r_cc[2], r_np[2], rtol=1e-11, atol=1e-12)


def test_backward_agrees_with_numpy_oracle():
    x = _case(4)
    _, idx, O, m, l = oracle.dsa_forward(x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], x["k"],
                                         x["scale"], x["d_v"])
    dq, dkv = oracle.sparse_attn_bwd(x["q"], x["kv"], idx, O, x["dO"], m, l, x["scale"], x["d_v"])
    dq2, dkv2 = cpp.sparse_attn_bwd(x["q"], x["kv"], idx, O, x["dO"], m, l, x["scale"], x["d_v"],
                                    threads=5)
    np.testing.assert_allclose(dq2, dq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dkv2, dkv, rtol=1e-10, atol=1e-12)
    kl = oracle.indexer_kl_loss(x["q"], x["kv"], idx, m, l, x["scale"], x["q_I"], x["k_I"], x["w"])
    kl2 = cpp.indexer_kl_loss(x["q"], x["kv"], idx, m, l, x["scale"], x["q_I"], x["k_I"], x["w"],
                              threads=5)
    assert abs(kl2[0] - kl[0]) <= 1e-12 * max(1.0, abs(kl[0]))
    for a, b in zip(kl2[1:], kl[1:]):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_hand_fixtures(golden):
    g = golden("indexer_hand.json")
    I = cpp.indexer_scores(np.array(g["q_I"]), np.array(g["k_I"]), np.array(g["w"]), np.array(g["pos"]))
    want = np.array([[[v if v is not None else -np.inf for v in r] for r in b] for b in g["expected_I"]])
    assert np.array_equal(np.isinf(I), np.isinf(want))
    np.testing.assert_allclose(I[np.isfinite(want)], want[np.isfinite(want)], atol=1e-15)

    t = golden("topk_hand.json")
    sc = np.array(t["scores"], dtype=np.float32)[None, None]
    for case in t["cases"]:
        got = cpp.topk_select(sc, np.array([[case["pos"]]]), case["k"])[0, 0].tolist()
        assert got == case["expected"], case["why"]

    a = golden("attention_hand.json")
    O, m, l = cpp.sparse_attn_fwd(np.array(a["q"]), np.array(a["kv"]), np.array(a["idx"]), a["scale"],
                                  a["d_v"])
    np.testing.assert_allclose(O, np.array(a["expected_O"]), atol=1e-14)
    np.testing.assert_allclose(m, np.array(a["expected_m"]), atol=1e-15)
    np.testing.assert_allclose(l, np.array(a["expected_l"]), atol=1e-15)

    for name in ("kl_loss_hand.json", "kl_loss_hand_2heads.json"):
        k = golden(name)
        arr = lambda n: np.array(k[n])
        loss, dq_I, dk_I, dw = cpp.indexer_kl_loss(arr("q"), arr("kv"), arr("idx"), arr("m"), arr("l"),
                                                   k["scale"], arr("q_I"), arr("k_I"), arr("w"))
        assert abs(loss - k["expected_loss"]) < 1e-14, name
        np.testing.assert_allclose(dw, arr("expected_dw"), atol=1e-15)
        np.testing.assert_allclose(dq_I, arr("expected_dq_I"), atol=1e-15)
        np.testing.assert_allclose(dk_I, arr("expected_dk_I"), atol=1e-15)


def test_dense_limit_equals_causal_sdpa_and_autograd():
    B, S, H, d_qk, d_v, scale = 2, 19, 3, 10, 6, 0.37
    rng = np.random.default_rng(11)
    q = rng.standard_normal((B, S, H, d_qk))
    kv = rng.standard_normal((B, S, d_qk))
    dO = rng.standard_normal((B, S, H, d_v))
    idx = np.full((B, S, S + 2), -1, dtype=np.int32)
    for t in range(S):
        idx[:, t, :t + 1] = np.arange(t + 1)
    O, m, l = cpp.sparse_attn_fwd(q, kv, idx, scale, d_v, threads=4)
    qt = torch.from_numpy(q).requires_grad_(True)
    kvt = torch.from_numpy(kv).requires_grad_(True)
    k_ = kvt[:, None].expand(B, H, S, d_qk)
    ref = F.scaled_dot_product_attention(qt.transpose(1, 2), k_, k_[..., :d_v], is_causal=True,
                                         scale=scale).transpose(1, 2)
    np.testing.assert_allclose(O, ref.detach().numpy(), rtol=1e-12, atol=1e-12)
    ref.backward(torch.from_numpy(dO))
    dq, dkv = cpp.sparse_attn_bwd(q, kv, idx, O, dO, m, l, scale, d_v, threads=4)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dkv, kvt.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_kl_finite_differences():
    rng = np.random.default_rng(31)
    S, H, d_qk, H_I, d_I, k, scale = 14, 3, 6, 2, 4, 5, 0.5
    q = rng.standard_normal((1, S, H, d_qk))
    kv = rng.standard_normal((1, S, d_qk))
    qI = rng.standard_normal((1, S, H_I, d_I))
    kI = rng.standard_normal((1, S, d_I))
    w = rng.standard_normal((1, S, H_I))
    idx = cpp.topk_select(rng.standard_normal((1, S, S)), cpp.positions(1, S), k)
    _, m, l = cpp.sparse_attn_fwd(q, kv, idx, scale, 1)
    loss, dqI, dkI, dw = cpp.indexer_kl_loss(q, kv, idx, m, l, scale, qI, kI, w)
    f = lambda: cpp.indexer_kl_loss(q, kv, idx, m, l, scale, qI, kI, w, threads=1)[0]
    eps = 1e-6
    picks = [(0, 3, 1, 2), (0, 9, 0, 0), (0, 13, 1, 3)]
    for arr, grad in ((qI, dqI), (kI, dkI), (w, dw)):
        for full in picks:
            i = full[: arr.ndim]
            old = arr[i]
            arr[i] = old + eps
            fp = f()
            arr[i] = old - eps
            fm = f()
            arr[i] = old
            assert abs((fp - fm) / (2 * eps) - grad[i]) < 1e-7, i


def test_topk_ties_signed_zero_and_threads():
    rng = np.random.default_rng(5)
    S = 300
    sc = rng.integers(-3, 4, size=(1, S, S)).astype(np.float32)   # heavy ties
    sc[0, :, ::7] = -0.0
    pos = cpp.positions(1, S)
    a = cpp.topk_select(sc, pos, 17, threads=1)
    b = cpp.topk_select(sc, pos, 17, threads=8)
    assert np.array_equal(a, b)
    assert np.array_equal(a, oracle.topk_select(sc, pos, 17))
