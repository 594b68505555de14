"""Batched calls (BSND layout, B = 2): every query row attends its own
sequence's keys [HP-CP, layouts BSND / TND], so a B = 2 call must give, per
batch entry, what the oracle gives for that sequence and what a B = 1 call on
that sequence alone gives (bit for bit: rows and keys are independent of the
other batch entry)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (DEV, FP32_TOL, bf16_close, empty_outputs, lib, near_tie_violations, np64,
                      params)

pytestmark = pytest.mark.gpu


def _forward(wl, x):
    dsa = lib()
    p = params(dsa, wl)
    o = empty_outputs(wl, wl["S"], torch.float32 if wl["dtype"] == "fp32" else torch.bfloat16)
    ws = torch.empty(max(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD), 16), dtype=torch.uint8,
                     device=DEV)
    dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], o["idx"], o["out"], o["m"], o["l"], ws)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    return o


def test_fp32_batch2_against_oracle():
    wl = dict(synth.TINY, B=2)
    x = synth.make_inputs(wl)
    sc, idx, O, m, l = oracle.dsa_forward(x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], wl["topk"],
                                          wl["scale"], wl["d_v"])
    o = _forward(wl, {n: v.to(DEV) for n, v in x.items()})
    gi = o["idx"].cpu().numpy()
    for b in range(2):
        assert near_tie_violations(gi[b], idx[b], sc[b], wl["topk"]) == []
    same = np.all(gi == idx, axis=2)          # rows whose index sets match exactly
    assert same.mean() > 0.9
    assert np.abs(np64(o["out"])[same] - O[same]).max() < FP32_TOL
    assert np.abs(np64(o["m"])[same] - m[same]).max() < FP32_TOL
    assert np.abs(np64(o["l"])[same] - l[same]).max() < FP32_TOL


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_batch2_equals_single_sequences(dtype):
    wl = dict(synth.TINY, B=2) if dtype == "fp32" else dict(synth.v32(448, "dsv32_S448"), topk=200, B=2)
    x = {n: v.to(DEV) for n, v in synth.make_inputs(wl).items()}
    both = _forward(wl, x)
    one = dict(wl, B=1)
    for b in range(2):
        ob = _forward(one, {n: v[b:b + 1].contiguous() for n, v in x.items()})
        for key in ("idx", "out", "m", "l"):
            assert torch.equal(both[key][b:b + 1], ob[key]), (b, key)


def test_bf16_batch2_attention_against_oracle():
    wl = dict(synth.v32(448, "dsv32_S448"), topk=200, B=2)
    x = synth.make_inputs(wl)
    pos = oracle.positions(2, wl["S"])
    sc = oracle.indexer_scores(x["q_I"], x["k_I"], x["w"], pos)
    ridx = oracle.topk_select(sc, pos, wl["topk"])
    O, m, l = oracle.sparse_attn_fwd(x["q"], x["kv"], ridx, wl["scale"], wl["d_v"])
    dsa = lib()
    p = params(dsa, wl)
    o = empty_outputs(wl, wl["S"], torch.bfloat16)
    dsa.sparse_attn_fwd(p, x["q"].to(DEV), x["kv"].to(DEV), torch.as_tensor(ridx, device=DEV),
                        o["out"], o["m"], o["l"])
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    ok, ma, mr = bf16_close(np64(o["out"]), O)
    assert ok, (ma, mr)
    assert np.abs(np64(o["m"]) - m).max() < 1e-4


def test_auto_wave_is_whole_indexer_rounds():
    # the forward's score ring holds one wave; its auto size is a multiple of
    # 4 rows x the SM count (one four-row indexer CTA per SM per round) when
    # the 256 MB budget allows it, the whole call when that is shorter, and
    # 1024 rows when not even one round fits
    dsa = lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for S in (4096, 16384, 32768, 65536, 131072):
        wl = dict(synth.v32(S, f"dsv32_S{S}"))
        p = params(dsa, wl)
        w = dsa.wave_rows(p)
        budget = (256 << 20) // (4 * S)
        if budget >= S:
            assert w == S
        elif budget >= 4 * sms:
            assert w % (4 * sms) == 0 and w <= budget and w + 4 * sms > budget, (S, w)
        else:
            assert w == 1024
