"""Exact-arithmetic (fp32) path on the tiny DSA configuration (S=256, 8 heads,
d_qk=80, d_v=64, indexer 4x32, top-32), against the fp64 oracle: max-abs 1e-5."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, FP32_TOL, empty_outputs, lib, near_tie_violations, np64, params

pytestmark = pytest.mark.gpu

WL = synth.TINY


@pytest.fixture(scope="module")
def case():
    x = synth.make_inputs(WL)
    sc, idx, O, m, l = oracle.dsa_forward(x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], WL["topk"],
                                          WL["scale"], WL["d_v"])
    return x, dict(scores=sc, idx=idx, O=O, m=m, l=l)


def test_indexer_scores(case):
    dsa = lib()
    x, ref = case
    S = WL["S"]
    p = params(dsa, WL)
    sc = torch.empty(S, S, device=DEV)
    g = {k: v.to(DEV) for k, v in x.items()}
    dsa.indexer_scores(p, g["q_I"], g["k_I"], g["w"], 0, S, sc)
    torch.cuda.synchronize()
    got = np64(sc)
    exp = ref["scores"][0]
    fin = np.isfinite(exp)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - exp[fin]).max() < FP32_TOL


def test_attention_on_oracle_indices(case):
    dsa = lib()
    x, ref = case
    S = WL["S"]
    p = params(dsa, WL)
    o = empty_outputs(WL, S, torch.float32)
    idx = torch.as_tensor(ref["idx"], device=DEV)
    dsa.sparse_attn_fwd(p, x["q"].to(DEV), x["kv"].to(DEV), idx, o["out"], o["m"], o["l"])
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    assert np.abs(np64(o["out"]) - ref["O"]).max() < FP32_TOL
    assert np.abs(np64(o["m"]) - ref["m"]).max() < FP32_TOL
    assert np.abs(np64(o["l"]) - ref["l"]).max() < FP32_TOL


def test_forward_end_to_end(case):
    dsa = lib()
    x, ref = case
    S, k = WL["S"], WL["topk"]
    p = params(dsa, WL)
    o = empty_outputs(WL, S, torch.float32)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) // 4, device=DEV)
    g = {n: v.to(DEV) for n, v in x.items()}
    dsa.forward(p, g["q_I"], g["k_I"], g["w"], g["q"], g["kv"], o["idx"], o["out"], o["m"], o["l"], ws)
    torch.cuda.synchronize()
    gi = o["idx"].cpu().numpy()[0]
    assert near_tie_violations(gi, ref["idx"][0], ref["scores"][0], k) == []
    # every row: the oracle's attention over the GPU's own index sets (equal
    # to the oracle's own sets up to near-tied keys, checked above)
    O, m, l = oracle.sparse_attn_fwd(x["q"], x["kv"], gi[None], WL["scale"], WL["d_v"])
    assert np.abs(np64(o["out"]) - O).max() < FP32_TOL
    assert np.abs(np64(o["m"]) - m).max() < FP32_TOL
    assert np.abs(np64(o["l"]) - l).max() < FP32_TOL


def test_cp_shards_bit_identical(case):
    dsa = lib()
    x, _ = case
    S, k = WL["S"], WL["topk"]
    g = {n: v.to(DEV) for n, v in x.items()}

    def run(rows, **kw):
        n = len(rows)
        p = params(dsa, WL, S_q=n, **kw)
        o = empty_outputs(WL, n, torch.float32)
        ws = torch.empty(max(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) // 4, 4), device=DEV)
        dsa.forward(p, g["q_I"][:, rows].contiguous(), g["k_I"], g["w"][:, rows].contiguous(),
                    g["q"][:, rows].contiguous(), g["kv"], o["idx"], o["out"], o["m"], o["l"], ws)
        torch.cuda.synchronize()
        return o

    full = run(list(range(S)))
    off = run(list(range(64, 128)), q_row_offset=64)
    ht_rows = synth.head_tail_rows(S, 4, 1)
    keep = torch.as_tensor(ht_rows, device=DEV)
    ht = run(ht_rows.tolist(), q_row_index=keep)
    for part, rows in ((off, list(range(64, 128))), (ht, ht_rows.tolist())):
        for key in ("idx", "out", "m", "l"):
            assert torch.equal(part[key], full[key][:, rows]), key


def test_backward(case):
    dsa = lib()
    x, ref = case
    S, H, d_qk, d_v = WL["S"], WL["H"], WL["d_qk"], WL["d_v"]
    dO = synth.normal((1, S, H, d_v), "dO", 0, 1.0, torch.float32)
    dq_r, dkv_r = oracle.sparse_attn_bwd(x["q"], x["kv"], ref["idx"], ref["O"], dO, ref["m"],
                                         ref["l"], WL["scale"], d_v)
    p = params(dsa, WL)
    f32 = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.float32, device=DEV).contiguous()
    idx = torch.as_tensor(ref["idx"], device=DEV)
    dq = torch.empty(1, S, H, d_qk, device=DEV)
    dkv = torch.zeros(1, S, d_qk, device=DEV)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_ATTN_BWD) // 4, device=DEV)
    dsa.sparse_attn_bwd(p, x["q"].to(DEV), x["kv"].to(DEV), idx, f32(ref["O"]), dO.to(DEV),
                        f32(ref["m"]), f32(ref["l"]), dq, dkv, ws)
    torch.cuda.synchronize()
    assert np.abs(np64(dq) - dq_r).max() < FP32_TOL
    assert np.abs(np64(dkv) - dkv_r).max() < FP32_TOL

    loss_r, dqI_r, dkI_r, dw_r = oracle.indexer_kl_loss(x["q"], x["kv"], ref["idx"], ref["m"],
                                                         ref["l"], WL["scale"], x["q_I"], x["k_I"],
                                                         x["w"])
    loss = torch.zeros(1, device=DEV)
    dqI = torch.empty_like(x["q_I"], device=DEV)
    dkI = torch.zeros_like(x["k_I"], device=DEV)
    dw = torch.empty_like(x["w"], device=DEV)
    dsa.indexer_kl_loss_bwd(p, x["q"].to(DEV), x["kv"].to(DEV), x["q_I"].to(DEV), x["k_I"].to(DEV),
                            x["w"].to(DEV), idx, f32(ref["m"]), f32(ref["l"]), loss, dqI, dkI, dw,
                            torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_KL_BWD) // 4, device=DEV))
    torch.cuda.synchronize()
    assert abs(float(loss) - loss_r) < FP32_TOL * max(1.0, abs(loss_r))
    assert np.abs(np64(dqI) - dqI_r).max() < FP32_TOL
    assert np.abs(np64(dkI) - dkI_r).max() < FP32_TOL
    assert np.abs(np64(dw) - dw_r).max() < FP32_TOL
