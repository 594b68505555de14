"""Fused Lightning Indexer + streaming top-k (dsa_indexer_topk and dsa_forward
with DSA_FLAG_FUSED_TOPK) against the unfused path on the same inputs.

The fused kernel computes every score with the unfused indexer's arithmetic
and keeps all keys at or above a running threshold that never exceeds the
row's k-th largest key, so its indices must equal dsa_indexer_scores followed
by dsa_topk bit for bit (the unfused top-k is itself pinned bit-exactly to
the oracle's selection in test_gpu_topk.py).  The adversarial cases make
every key a candidate (scores rising with position) or every key equal."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import DEV, lib, params

pytestmark = pytest.mark.gpu


def _indexer_inputs(wl, S_q, seed=0):
    g = lambda shape, nm, sc: synth.normal(shape, nm, seed, sc, torch.bfloat16, DEV)
    B, S = wl["B"], wl["S"]
    return dict(q_I=g((B, S_q, wl["H_I"], wl["d_I"]), "q_I", 1.0),
                k_I=g((B, S, wl["d_I"]), "k_I", 1.0),
                w=g((B, S_q, wl["H_I"]), "w", 1.0 / 8.0))


def _both(dsa, p, x, row_begin, rows):
    """(fused idx, unfused idx) for flattened rows [row_begin, row_begin+rows)."""
    k, S_k = p.topk, p.S_k
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_INDEXER_TOPK), dtype=torch.uint8, device=DEV)
    fused = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    dsa.indexer_topk(p, x["q_I"], x["k_I"], x["w"], row_begin, rows, fused, ws)
    sc = torch.empty(rows, S_k, device=DEV)
    dsa.indexer_scores(p, x["q_I"], x["k_I"], x["w"], row_begin, rows, sc)
    ref = torch.full((rows, k), -9, dtype=torch.int32, device=DEV)
    dsa.topk(p, sc, row_begin, rows, ref)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    return fused.cpu().numpy(), ref.cpu().numpy()


def _assert_equal(fused, ref):
    bad = np.nonzero((fused != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:4]}"


def test_fused_equals_unfused_small_ragged():
    # S = 448, k = 200: rows with fewer than k causal keys, partial key blocks,
    # several waves (wave_rows = 96) so the candidate lists are reused
    dsa = lib()
    wl = dict(synth.v32(448, "dsv32_S448"), topk=200)
    p = params(dsa, wl, wave_rows=96)
    x = _indexer_inputs(wl, wl["S"])
    _assert_equal(*_both(dsa, p, x, 0, wl["S"]))


def test_fused_equals_unfused_32k_rows():
    # S = 32768, top-2048: the last 608 rows (the longest) and rows around k
    dsa = lib()
    wl = synth.WORKLOADS["dsv32_S32768"]
    S = wl["S"]
    p = params(dsa, wl)
    x = _indexer_inputs(wl, S)
    _assert_equal(*_both(dsa, p, x, S - 608, 608))
    _assert_equal(*_both(dsa, p, x, 2040, 64))


def test_fused_every_key_a_candidate():
    # scores rise with position (k_I[s] = ramp * e0, q_I = e0, w > 0): the
    # running threshold never drops a key before the row ends, and bf16
    # rounding of the ramp makes runs of equal scores (ties broken by index)
    dsa = lib()
    S, k = 4096, 256
    wl = dict(synth.v32(S, "ramp"), topk=k)
    p = params(dsa, wl)
    q_I = torch.zeros(1, S, 64, 128, dtype=torch.bfloat16, device=DEV)
    q_I[..., 0] = 1.0
    k_I = torch.zeros(1, S, 128, dtype=torch.bfloat16, device=DEV)
    k_I[0, :, 0] = (torch.arange(S, device=DEV, dtype=torch.float32) / S).to(torch.bfloat16)
    w = torch.full((1, S, 64), 1.0 / 64, dtype=torch.bfloat16, device=DEV)
    x = dict(q_I=q_I, k_I=k_I, w=w)
    fused, ref = _both(dsa, p, x, 0, S)
    _assert_equal(fused, ref)
    # the last row keeps the k largest positions' scores
    assert fused[-1, -1] == S - 1


def test_fused_all_scores_equal():
    # k_I = 0: every visible score is 0, so each row takes its first k positions
    dsa = lib()
    S, k = 2048, 128
    wl = dict(synth.v32(S, "flat"), topk=k)
    p = params(dsa, wl)
    x = _indexer_inputs(wl, S)
    x["k_I"] = torch.zeros_like(x["k_I"])
    fused, ref = _both(dsa, p, x, 0, S)
    _assert_equal(fused, ref)
    assert (fused[S - 1] == np.arange(k)).all()


def test_forward_fused_flag_equals_plain():
    # dsa_forward with DSA_FLAG_FUSED_TOPK: same indices, and so the same
    # attention outputs, as the plain forward (S = 4096, top-2048)
    dsa = lib()
    wl = synth.WORKLOADS["dsv32_S4096"]
    S = wl["S"]
    x = synth.make_inputs(wl, device=DEV)
    res = []
    for flags in (0, dsa.DSA_FLAG_FUSED_TOPK):
        p = params(dsa, wl, flags=flags)
        ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD), dtype=torch.uint8, device=DEV)
        idx = torch.empty(1, S, wl["topk"], dtype=torch.int32, device=DEV)
        out = torch.empty(1, S, wl["H"], wl["d_v"], dtype=torch.bfloat16, device=DEV)
        m = torch.empty(1, S, wl["H"], device=DEV)
        l = torch.empty_like(m)
        dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], idx, out, m, l, ws)
        torch.cuda.synchronize()
        assert dsa.get_status() == 0
        res.append((idx, out, m, l))
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_fused_batches_and_head_tail_rows():
    # B = 2 (rows of both batches in one call, each against its own keys) and
    # a head-tail context-parallel shard given by q_row_index
    dsa = lib()
    S, k = 2048, 256
    wl = dict(synth.v32(S, "b2"), B=2, topk=k)
    x = _indexer_inputs(wl, S, seed=3)
    p = params(dsa, wl, B=2)
    _assert_equal(*_both(dsa, p, x, 0, 2 * S))
    _assert_equal(*_both(dsa, p, x, S - 100, 300))       # straddles the batch boundary
    rows = np.r_[0:256, S - 256:S].astype(np.int32)      # head and tail of one sequence
    ridx = torch.as_tensor(rows, device=DEV)
    wl1 = dict(synth.v32(S, "ht"), topk=k)
    x1 = _indexer_inputs(wl1, S, seed=4)
    sel = torch.as_tensor(rows, dtype=torch.long, device=DEV)
    x1 = dict(q_I=x1["q_I"][:, sel].contiguous(), k_I=x1["k_I"], w=x1["w"][:, sel].contiguous())
    p1 = params(dsa, wl1, S_q=len(rows), q_row_index=ridx)
    _assert_equal(*_both(dsa, p1, x1, 0, len(rows)))
