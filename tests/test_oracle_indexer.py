"""Pins for the oracle's Lightning Indexer (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import indexer_scores, positions


def test_hand_example(golden):
    g = golden("indexer_hand.json")
    I = indexer_scores(np.array(g["q_I"]), np.array(g["k_I"]), np.array(g["w"]), np.array(g["pos"]))
    exp = g["expected_I"][0][0]
    assert I[0, 0, 0] == exp[0] and I[0, 0, 1] == exp[1]
    assert np.isneginf(I[0, 0, 2])


def test_single_head_unit_weight_is_relu_gemm():
    # H_I = 1 and w = 1 reduce the indexer to ReLU of a plain matrix product.
    rng = np.random.default_rng(1)
    S, d = 37, 9
    qI = rng.standard_normal((1, S, 1, d))
    kI = rng.standard_normal((1, S, d))
    w = np.ones((1, S, 1))
    I = indexer_scores(qI, kI, w, positions(1, S))
    ref = torch.relu(torch.from_numpy(qI[0, :, 0]) @ torch.from_numpy(kI[0]).T)
    mask = torch.triu(torch.ones(S, S, dtype=torch.bool), 1)
    ref = ref.masked_fill(mask, float("-inf")).numpy()
    np.testing.assert_allclose(I[0], ref, rtol=1e-13, atol=1e-13)


def test_brute_force_loops():
    rng = np.random.default_rng(2)
    B, S, H_I, d = 2, 11, 3, 5
    qI = rng.standard_normal((B, S, H_I, d))
    kI = rng.standard_normal((B, S, d))
    w = rng.standard_normal((B, S, H_I))
    pos = positions(B, S)
    I = indexer_scores(qI, kI, w, pos)
    for b in range(B):
        for t in range(S):
            for s in range(S):
                if s > t:
                    assert np.isneginf(I[b, t, s])
                    continue
                acc = 0.0
                for j in range(H_I):
                    dot = sum(qI[b, t, j, e] * kI[b, s, e] for e in range(d))
                    acc += w[b, t, j] * (dot if dot > 0 else 0.0)
                assert abs(I[b, t, s] - acc) < 1e-12


def test_heads_independent_and_linear_in_w():
    rng = np.random.default_rng(3)
    S, H_I, d = 16, 4, 6
    qI = rng.standard_normal((1, S, H_I, d))
    kI = rng.standard_normal((1, S, d))
    w = rng.standard_normal((1, S, H_I))
    pos = positions(1, S)
    full = indexer_scores(qI, kI, w, pos)
    parts = sum(indexer_scores(qI[:, :, j:j + 1], kI, w[:, :, j:j + 1], pos) for j in range(H_I))
    fin = np.isfinite(full)
    np.testing.assert_allclose(full[fin], parts[fin], rtol=1e-12, atol=1e-12)
    perm = rng.permutation(H_I)
    np.testing.assert_allclose(indexer_scores(qI[:, :, perm], kI, w[:, :, perm], pos)[fin], full[fin],
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(indexer_scores(qI, kI, 3.0 * w, pos)[fin], 3.0 * full[fin], rtol=1e-12)
