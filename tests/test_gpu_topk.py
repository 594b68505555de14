"""GPU top-k against the oracle on the same fp32 score tensor: bit-exact."""
import numpy as np
import pytest
import torch

import synth
from oracle import topk_select
from gpu_util import DEV, lib

pytestmark = pytest.mark.gpu


def _run(dsa, scores, pos, k):
    """scores [R, S_k] (host fp32), pos [R] global positions -> GPU idx [R, k]."""
    R, S_k = scores.shape
    ridx = torch.as_tensor(np.asarray(pos, dtype=np.int32), device=DEV)
    p = dsa.make_params(B=1, S_q=R, S_k=S_k, H=1, d_qk=8, d_v=8, H_I=1, d_I=8, topk=k, scale=1.0,
                        dtype="fp32", q_row_index=ridx)
    sc = torch.as_tensor(scores, device=DEV).contiguous()
    idx = torch.full((R, k), -7, dtype=torch.int32, device=DEV)
    dsa.topk(p, sc, 0, R, idx)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    return idx.cpu().numpy()


def _check(dsa, scores, pos, k):
    got = _run(dsa, scores, pos, k)
    ref = topk_select(scores[None], np.asarray(pos)[None], k)[0]
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first row {bad[:3]}"


def test_hand_example(golden):
    dsa = lib()
    g = golden("topk_hand.json")
    row = np.array(g["scores"], dtype=np.float32)
    for c in g["cases"]:
        got = _run(dsa, row[None], [c["pos"]], c["k"])[0].tolist()
        assert got == c["expected"], c["why"]


@pytest.mark.parametrize("k", [1, 17, 64, 299, 400])
def test_ties_and_signed_zero(k):
    dsa = lib()
    rng = np.random.default_rng(k)
    S = 300
    sc = rng.integers(-4, 5, size=(S, S)).astype(np.float32)
    z = sc == 0
    sc[z] = np.where(rng.random(z.sum()) < 0.5, -0.0, 0.0)
    _check(dsa, sc, np.arange(S), k)


@pytest.mark.parametrize("S_k,k,rows", [(1001, 100, 200), (4096, 2048, 512), (32768, 2048, 320),
                                        (40000, 2048, 24)])
def test_random_rows(S_k, k, rows):
    # 4096..32768: register-resident rows (more rows than SMs, so CTAs take
    # several rows each); 40000: streaming variant; 1001: rows
    # not 16-byte aligned (scalar loads)
    dsa = lib()
    sc = synth.normal((rows, S_k), 7, seed=1, dtype=torch.float32).numpy() * 8.0
    rng = np.random.default_rng(S_k)
    pos = rng.integers(0, S_k, size=rows)
    pos[:4] = [S_k - 1, k - 1, k, 0]
    _check(dsa, sc, pos, k)


def test_heavy_ties_long_row():
    # few distinct values: the radix passes end with large equal-key groups
    dsa = lib()
    rng = np.random.default_rng(3)
    S_k, k = 32768, 2048
    sc = rng.integers(0, 3, size=(8, S_k)).astype(np.float32)
    sc[1] = 1.0
    sc[2, ::2] = -0.0
    _check(dsa, sc, [S_k - 1, S_k - 1, S_k - 1, 5000, 30000, 2047, 2048, 12345], k)


@pytest.mark.parametrize("S_k", [4096, 8192, 16384])
@pytest.mark.parametrize("values", [1, 3, 1000, 0])
def test_sized_blocks_offset_rows(S_k, values):
    # rows addressed by offset (no q_row_index), so the launch sizes its
    # blocks by the longest row: up to 4096 keys the 256-thread form (16 keys
    # per thread), up to 8192 1024-thread blocks of two 512-thread groups
    # with a row each (16 keys per thread), up to 16384 the same with 32.
    # With one value the threshold's bin holds every key (the passes run over
    # registers once it exceeds the candidate list: 4096 entries, 2048 per
    # group), with 3 a third of them, with 1000 a few dozen to a few hundred,
    # with 0 normal scores
    dsa = lib()
    k, rows = 2048, 96
    r0 = S_k - rows
    p = dsa.make_params(B=1, S_q=S_k, S_k=S_k, H=1, d_qk=8, d_v=8, H_I=1, d_I=8, topk=k, scale=1.0,
                        dtype="fp32")
    rng = np.random.default_rng(values + S_k)
    if values:
        sc = rng.integers(0, values, size=(rows, S_k)).astype(np.float32)
    else:
        sc = synth.normal((rows, S_k), 11, seed=2, dtype=torch.float32).numpy() * 8.0
    got = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    dsa.topk(p, torch.as_tensor(sc, device=DEV), r0, rows, got)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    ref = topk_select(sc[None], np.arange(r0, r0 + rows)[None], k)[0]
    bad = np.nonzero((got.cpu().numpy() != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first row {bad[:3]}"


@pytest.mark.parametrize("values", [3, 0])
def test_offset_rows_across_16k_keys(values):
    # offset rows whose key counts run from 15985 to 16784: the launch sends
    # the rows of up to 16384 keys to the two-group form and the rest to the
    # one-row form, as two launches over the same output
    dsa = lib()
    S_k, k, rows = 32768, 2048, 800
    r0 = 16384 - 400
    p = dsa.make_params(B=1, S_q=S_k, S_k=S_k, H=1, d_qk=8, d_v=8, H_I=1, d_I=8, topk=k, scale=1.0,
                        dtype="fp32")
    rng = np.random.default_rng(values + 17)
    if values:
        sc = rng.integers(0, values, size=(rows, S_k)).astype(np.float32)
    else:
        sc = synth.normal((rows, S_k), 13, seed=4, dtype=torch.float32).numpy() * 8.0
    got = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    dsa.topk(p, torch.as_tensor(sc, device=DEV), r0, rows, got)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    ref = topk_select(sc[None], np.arange(r0, r0 + rows)[None], k)[0]
    bad = np.nonzero((got.cpu().numpy() != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first row {bad[:3]}"
