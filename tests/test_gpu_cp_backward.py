"""Context-parallel contract of the backward: the per-key gradients (dKV,
dk_I) and the loss that query-row shards accumulate sum to the unsharded
result, and the per-row gradients (dQ, dq_I, dw) of a shard equal those rows
of the unsharded call.

[HP-CP] head-tail placement (rank r of CP ranks holds row chunks r and
2*CP-1-r); [DSA-32K] SFAG / SLIG accumulate dKV and dk_I over the query rows
of the call.  Two ranks are emulated on one GPU by two calls on disjoint row
sets writing into the same accumulators."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, bf16_close, lib, np64, params

pytestmark = pytest.mark.gpu


def _inputs(wl):
    dsa = lib()
    S = wl["S"]
    x = synth.make_inputs(wl, device=DEV, with_dout=True)
    p = params(dsa, wl)
    idx = torch.empty(1, S, wl["topk"], dtype=torch.int32, device=DEV)
    out = torch.empty(1, S, wl["H"], wl["d_v"], dtype=torch.bfloat16, device=DEV)
    m = torch.empty(1, S, wl["H"], device=DEV)
    l = torch.empty_like(m)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD), dtype=torch.uint8, device=DEV)
    dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], idx, out, m, l, ws)
    return x, idx, out, m, l


def _backward(wl, x, idx, out, m, l, rows, acc):
    """dsa_backward on the query rows `rows` (global positions), accumulating
    dkv / dk_I / loss into acc; returns the per-row outputs."""
    dsa = lib()
    r = torch.as_tensor(np.asarray(rows), dtype=torch.long, device=DEV)
    n = len(rows)
    p = params(dsa, wl, S_q=n, q_row_index=torch.as_tensor(np.asarray(rows, np.int32), device=DEV))
    sel = lambda t: t[:, r].contiguous()
    dq = torch.empty(1, n, wl["H"], wl["d_qk"], dtype=torch.bfloat16, device=DEV)
    dqI = torch.empty(1, n, wl["H_I"], wl["d_I"], dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(1, n, wl["H_I"], device=DEV)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_BACKWARD), dtype=torch.uint8, device=DEV)
    dsa.backward(p, sel(x["q"]), x["kv"], sel(idx), sel(out), sel(x["dO"]), sel(m), sel(l),
                 sel(x["q_I"]), x["k_I"], sel(x["w"]), dq, acc["dkv"], acc["loss"], dqI, acc["dkI"],
                 dw, ws)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    return dict(dq=dq, dqI=dqI, dw=dw)


def _zeros(wl):
    S = wl["S"]
    return dict(dkv=torch.zeros(1, S, wl["d_qk"], device=DEV),
                dkI=torch.zeros(1, S, wl["d_I"], device=DEV), loss=torch.zeros(1, device=DEV))


def test_head_tail_shards_sum_to_unsharded():
    wl = dict(synth.v32(448, "dsv32_S448"), topk=200)
    S = wl["S"]
    x, idx, out, m, l = _inputs(wl)
    full = _zeros(wl)
    f = _backward(wl, x, idx, out, m, l, list(range(S)), full)
    # CP = 2, four chunks of 112 rows: rank 0 holds chunks 0 and 3, rank 1 chunks 1 and 2
    c = S // 4
    shards = [list(range(0, c)) + list(range(3 * c, S)), list(range(c, 3 * c))]
    part = _zeros(wl)
    for rows in shards:
        g = _backward(wl, x, idx, out, m, l, rows, part)
        for key in ("dq", "dqI", "dw"):   # rows are independent: bit for bit
            assert torch.equal(g[key][0], f[key][0, rows]), key
    # per-key sums: the same terms added in another order (fp32 atomics)
    for key in ("dkv", "dkI"):
        ref = full[key].double()
        err = (part[key].double() - ref).abs().max().item()
        assert err <= 1e-5 * max(ref.abs().max().item(), 1.0), (key, err)
    assert abs(part["loss"].item() - full["loss"].item()) <= 1e-5 * abs(full["loss"].item())
    # and the shard sums equal the oracle's unsharded backward of the same
    # forward results (idx, out, m, l), at the bf16 agreement rule
    xc = {n: v.cpu() for n, v in x.items()}
    gidx = idx.cpu().numpy()
    Od, md, ld = np64(out), np64(m), np64(l)
    _, dkv_r = oracle.sparse_attn_bwd(xc["q"], xc["kv"], gidx, Od, xc["dO"], md, ld, wl["scale"],
                                      wl["d_v"])
    loss_r, _, dkI_r, _ = oracle.indexer_kl_loss(xc["q"], xc["kv"], gidx, md, ld, wl["scale"],
                                                 xc["q_I"], xc["k_I"], xc["w"])
    for key, ref in (("dkv", dkv_r), ("dkI", dkI_r)):
        ok, ma, mr = bf16_close(np64(part[key]), ref)
        assert ok, (key, ma, mr)
    assert abs(part["loss"].item() - loss_r) <= 1e-3 * abs(loss_r), (part["loss"].item(), loss_r)
