"""Pins for the oracle's top-k selection (CPU only)."""
import numpy as np
import torch

from oracle import topk_select


def _brute(row, pos, k):
    n = pos + 1
    cand = sorted(range(n), key=lambda s: (-float(row[s]) if row[s] != 0 else 0.0, s))
    keep = sorted(cand[:min(k, n)])
    return keep + [-1] * (k - len(keep))


def test_hand_example(golden):
    g = golden("topk_hand.json")
    row = np.array(g["scores"], dtype=np.float32)
    for c in g["cases"]:
        sc = np.full((1, 1, row.size), np.nan, dtype=np.float32)
        sc[0, 0, :] = row
        got = topk_select(sc, np.array([[c["pos"]]]), c["k"])[0, 0].tolist()
        assert got == c["expected"], c["why"]


def test_brute_force_with_ties():
    rng = np.random.default_rng(5)
    S = 40
    for trial in range(20):
        k = int(rng.integers(1, 45))
        sc = rng.integers(-4, 5, size=(1, S, S)).astype(np.float32)
        sc[sc == 0] = np.where(rng.random(np.count_nonzero(sc == 0)) < 0.5, -0.0, 0.0)
        pos = np.arange(S)[None]
        got = topk_select(sc, pos, k)
        for t in range(S):
            assert got[0, t].tolist() == _brute(sc[0, t], t, k)


def test_matches_torch_topk_on_distinct_values():
    rng = np.random.default_rng(6)
    S, k = 300, 17
    sc = rng.standard_normal((2, S, S)).astype(np.float32)
    pos = np.broadcast_to(np.arange(S), (2, S))
    got = topk_select(sc, pos, k)
    for b in range(2):
        for t in range(k - 1, S):
            ref = torch.topk(torch.from_numpy(sc[b, t, :t + 1]), k).indices.sort().values.numpy()
            assert np.array_equal(got[b, t], ref)


def test_k_at_least_causal_length_is_prefix():
    S, k = 20, 25
    sc = np.random.default_rng(7).standard_normal((1, S, S)).astype(np.float32)
    got = topk_select(sc, np.arange(S)[None], k)
    for t in range(S):
        assert got[0, t].tolist() == list(range(t + 1)) + [-1] * (k - t - 1)


def test_masked_region_never_selected():
    S, k = 12, 4
    sc = np.zeros((1, S, S), dtype=np.float32)
    sc[0] = np.tril(np.ones((S, S))) + np.triu(np.full((S, S), 100.0), 1)
    got = topk_select(sc, np.arange(S)[None], k)
    for t in range(S):
        v = got[0, t][got[0, t] >= 0]
        assert (v <= t).all()
