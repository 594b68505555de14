"""bf16 tensor-core backward (sparse attention dQ / dKV and the indexer KL
loss gradients) at the DeepSeek-V3.2 head shapes against the fp64 oracle.

Both sides take the same forward results (the oracle's O rounded to bf16,
its softmax max / sum rounded to fp32) and the same index sets, so the
backward is checked on its own."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, bf16_close, lib, np64, params

pytestmark = pytest.mark.gpu


def _run_case(wl, rows, edit=None):
    """Oracle forward on `rows` (global positions) of workload `wl`, then the
    backward on both sides.  The q-side inputs are drawn for len(rows) rows;
    `edit(idx)` may rewrite the index sets in place before either side runs."""
    n, S, k = len(rows), wl["S"], wl["topk"]
    x = synth.make_inputs(wl, with_dout=True, S_q=n)
    pos = oracle.positions(1, n, q_row_index=np.asarray(rows))
    sc = oracle.indexer_scores(x["q_I"], x["k_I"], x["w"], pos)
    idx = oracle.topk_select(sc, pos, k)
    rng = np.random.default_rng(3)
    for r in range(0, n, 5):                 # shuffled slot order and -1 holes
        row = idx[0, r].copy()
        rng.shuffle(row)
        idx[0, r] = row
    if edit is not None:
        edit(idx)
    O, m, l = oracle.sparse_attn_fwd(x["q"], x["kv"], idx, wl["scale"], wl["d_v"])
    O16 = torch.as_tensor(O).to(torch.bfloat16)
    m32 = torch.as_tensor(m).float()
    l32 = torch.as_tensor(l).float()

    dsa = lib()
    p = params(dsa, wl, S_q=n)
    g = {nm: v.to(DEV) for nm, v in x.items()}
    gidx = torch.as_tensor(idx, device=DEV)
    dq = torch.empty(1, n, wl["H"], wl["d_qk"], dtype=torch.bfloat16, device=DEV)
    dkv = torch.zeros(1, S, wl["d_qk"], device=DEV)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_ATTN_BWD), dtype=torch.uint8, device=DEV)
    dsa.sparse_attn_bwd(p, g["q"], g["kv"], gidx, O16.to(DEV), g["dO"], m32.to(DEV), l32.to(DEV),
                        dq, dkv, ws)
    loss = torch.zeros(1, device=DEV)
    dqI = torch.empty(1, n, wl["H_I"], wl["d_I"], dtype=torch.bfloat16, device=DEV)
    dkI = torch.zeros(1, S, wl["d_I"], device=DEV)
    dw = torch.empty(1, n, wl["H_I"], device=DEV)
    ws2 = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_KL_BWD), dtype=torch.uint8, device=DEV)
    dsa.indexer_kl_loss_bwd(p, g["q"], g["kv"], g["q_I"], g["k_I"], g["w"], gidx, m32.to(DEV),
                            l32.to(DEV), loss, dqI, dkI, dw, ws2)
    # the same through dsa_backward (one call, shared recompute of P)
    f = dict(dq=torch.empty_like(dq), dkv=torch.zeros_like(dkv), loss=torch.zeros(1, device=DEV),
             dqI=torch.empty_like(dqI), dkI=torch.zeros_like(dkI), dw=torch.empty_like(dw))
    ws3 = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_BACKWARD), dtype=torch.uint8, device=DEV)
    dsa.backward(p, g["q"], g["kv"], gidx, O16.to(DEV), g["dO"], m32.to(DEV), l32.to(DEV), g["q_I"],
                 g["k_I"], g["w"], f["dq"], f["dkv"], f["loss"], f["dqI"], f["dkI"], f["dw"], ws3)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0

    Od = O16.double().numpy()
    dq_r, dkv_r = oracle.sparse_attn_bwd(x["q"], x["kv"], idx, Od, x["dO"], m32.double().numpy(),
                                         l32.double().numpy(), wl["scale"], wl["d_v"])
    kl_r = oracle.indexer_kl_loss(x["q"], x["kv"], idx, m32.double().numpy(),
                                  l32.double().numpy(), wl["scale"], x["q_I"], x["k_I"], x["w"])
    sep = dict(dq=(np64(dq), dq_r), dkv=(np64(dkv), dkv_r), loss=(float(loss), kl_r[0]),
               dqI=(np64(dqI), kl_r[1]), dkI=(np64(dkI), kl_r[2]), dw=(np64(dw), kl_r[3]))
    fused = dict(dq=(np64(f["dq"]), dq_r), dkv=(np64(f["dkv"]), dkv_r), loss=(float(f["loss"]), kl_r[0]),
                 dqI=(np64(f["dqI"]), kl_r[1]), dkI=(np64(f["dkI"]), kl_r[2]), dw=(np64(f["dw"]), kl_r[3]))
    # outputs written without atomics must match the separate calls bit for bit
    assert torch.equal(f["dq"], dq) and torch.equal(f["dqI"], dqI) and torch.equal(f["dw"], dw)
    return sep, fused


def _check(both):
    for res in both:
        _check_one(res)


def _check_one(res):
    for key in ("dq", "dkv", "dqI", "dkI", "dw"):
        got, ref = res[key]
        ok, ma, mr = bf16_close(got, ref)
        assert ok, (key, ma, mr)
    got, ref = res["loss"]
    assert abs(got - ref) <= 1e-3 * abs(ref), (got, ref)


def test_backward_small_ragged():
    # S = 448, k = 200: partial key tiles, rows with fewer than k causal keys
    wl = dict(synth.v32(448, "dsv32_S448"), topk=200)
    _check(_run_case(wl, list(range(448))))


def test_backward_train_shape_sampled_rows():
    # S = 16384, top-2048 (the training configuration): a shard of sampled
    # query rows against the full key side; dKV / dk_I sum over that shard
    wl = synth.WORKLOADS["dsv32_S16384_train"]
    S = wl["S"]
    rows = sorted(set([0, 1, 2047, 2048, 2049, 8191, S - 2, S - 1] +
                      np.random.default_rng(5).integers(0, S, 8).tolist()))
    _check(_run_case(wl, rows))


def test_backward_empty_rows_and_late_key_tiles():
    # k = 256 (two key tiles): some rows select nothing at all, others hold
    # their keys only in the second tile (the first tile is all holes), so
    # the dKV pass meets items with no valid tile and items whose first
    # valid tile is not the first one
    wl = dict(synth.v32(448, "dsv32_S448"), topk=256)

    def edit(idx):
        for r in range(idx.shape[1]):
            if r % 7 == 3:
                idx[0, r] = -1
            elif r % 7 == 5:
                keep = idx[0, r][idx[0, r] >= 0][:128]
                idx[0, r] = -1
                idx[0, r, 256 - keep.size:] = keep

    _check(_run_case(wl, list(range(448)), edit))


@pytest.mark.parametrize("B,wave,index", [(1, 100, False), (2, 160, False), (1, 24, True)])
def test_backward_in_row_passes(B, wave, index):
    # 0 < wave_rows < S_q: the bf16 backward runs in passes of at most
    # wave_rows rows of one batch, with a workspace for one pass.  Rows are
    # independent and dkv, dk_I and the loss accumulate, so dq, dq_I and dw
    # equal the one-pass call bit for bit and the accumulated outputs agree up
    # to the order of the atomic additions.  Cases: ragged last pass, two
    # batches, rows given by q_row_index (a context-parallel shard)
    dsa = lib()
    wl = dict(synth.v32(448, "passes"), topk=200, B=B)
    S = wl["S"]
    kw = {}
    n = S
    if index:
        rows = np.sort(np.random.default_rng(7).choice(S, 64, replace=False)).astype(np.int32)
        n = len(rows)
        kw = dict(S_q=n, q_row_index=torch.as_tensor(rows, device=DEV))
    x = {nm: v.to(DEV) for nm, v in synth.make_inputs(wl, with_dout=True, S_q=n).items()}
    p_one = params(dsa, wl, **kw)
    ws = torch.empty(dsa.workspace_size(p_one, dsa.DSA_CALL_FORWARD), dtype=torch.uint8, device=DEV)
    idx = torch.empty(B, n, wl["topk"], dtype=torch.int32, device=DEV)
    out = torch.empty(B, n, wl["H"], wl["d_v"], dtype=torch.bfloat16, device=DEV)
    m = torch.empty(B, n, wl["H"], device=DEV)
    l = torch.empty_like(m)
    dsa.forward(p_one, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], idx, out, m, l, ws)

    def run(p):
        r = dict(dq=torch.empty(B, n, wl["H"], wl["d_qk"], dtype=torch.bfloat16, device=DEV),
                 dkv=torch.zeros(B, S, wl["d_qk"], device=DEV), loss=torch.zeros(1, device=DEV),
                 dqI=torch.empty(B, n, wl["H_I"], wl["d_I"], dtype=torch.bfloat16, device=DEV),
                 dkI=torch.zeros(B, S, wl["d_I"], device=DEV),
                 dw=torch.empty(B, n, wl["H_I"], device=DEV))
        wsb = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_BACKWARD), dtype=torch.uint8, device=DEV)
        dsa.backward(p, x["q"], x["kv"], idx, out, x["dO"], m, l, x["q_I"], x["k_I"], x["w"],
                     r["dq"], r["dkv"], r["loss"], r["dqI"], r["dkI"], r["dw"], wsb)
        r["dq2"] = torch.empty_like(r["dq"])
        r["dkv2"] = torch.zeros_like(r["dkv"])
        wsa = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_ATTN_BWD), dtype=torch.uint8, device=DEV)
        dsa.sparse_attn_bwd(p, x["q"], x["kv"], idx, out, x["dO"], m, l, r["dq2"], r["dkv2"], wsa)
        torch.cuda.synchronize()
        assert dsa.get_status() == 0
        return r, wsb.numel()

    one, ws_one = run(p_one)
    parts, ws_parts = run(params(dsa, wl, wave_rows=wave, **kw))
    assert ws_parts < ws_one
    for key in ("dq", "dqI", "dw", "dq2"):
        assert torch.equal(parts[key], one[key]), key
    for key in ("dkv", "dkI", "dkv2"):
        ref = one[key]
        torch.testing.assert_close(parts[key], ref, rtol=1e-5, atol=1e-6 * float(ref.abs().max()))
    assert abs(float(parts["loss"]) - float(one["loss"])) <= 1e-5 * abs(float(one["loss"]))
