"""dsa_forward_static_ws, the forward for callers that cannot allocate device
memory (custom-operator hosts that provide only input/output buffers, loops
that must not call cudaMalloc): it must give the same results as dsa_forward
with a caller-provided workspace, on two calls in a row (the fixed ring keeps
the previous call's contents)."""
import pytest
import torch

import synth
from gpu_util import DEV, empty_outputs, lib, params

pytestmark = pytest.mark.gpu


def _compare(dsa, wl, x, p, S_q, rows):
    """dsa_forward (caller workspace) against dsa_forward_static_ws on the same
    rows, twice in a row; rows are independent and the kernels deterministic,
    so every output must be equal bit for bit."""
    sel = lambda t: t[:, rows].contiguous()
    q_I, w, q = sel(x["q_I"]), sel(x["w"]), sel(x["q"])
    ref = empty_outputs(wl, S_q, torch.bfloat16)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) // 4, device=DEV)
    dsa.forward(p, q_I, x["k_I"], w, q, x["kv"], ref["idx"], ref["out"], ref["m"], ref["l"], ws)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    for call in range(2):
        o = empty_outputs(wl, S_q, torch.bfloat16)
        dsa.forward_static_ws(p, q_I, x["k_I"], w, q, x["kv"], o["idx"], o["out"], o["m"], o["l"])
        torch.cuda.synchronize()
        assert dsa.get_status() == 0
        for key in ("idx", "out", "m", "l"):
            assert torch.equal(o[key], ref[key]), (call, key)


def test_static_ring_forward_matches_workspace_forward():
    # S = 4096: the fixed ring holds 2048 score rows, so the static path runs
    # two full waves where the workspace path runs one
    dsa = lib()
    wl = synth.WORKLOADS["dsv32_S4096"]
    S = wl["S"]
    x = synth.make_inputs(wl, device=DEV)
    _compare(dsa, wl, x, params(dsa, wl), S, torch.arange(S, device=DEV))


def test_static_ring_partial_last_wave():
    # a shard of 3000 rows at global positions 1096..4095: waves of 2048 and
    # 952 rows (the last one partial) against one workspace wave
    dsa = lib()
    wl = synth.WORKLOADS["dsv32_S4096"]
    x = synth.make_inputs(wl, device=DEV)
    n = 3000
    p = params(dsa, wl, S_q=n, q_row_offset=wl["S"] - n)
    _compare(dsa, wl, x, p, n, torch.arange(wl["S"] - n, wl["S"], device=DEV))


def test_static_ring_rejects_oversized_key_length():
    dsa = lib()
    p = dsa.make_params(B=1, S_q=4, S_k=3_000_000, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                        topk=16, scale=0.1, dtype="bf16")
    t = torch.empty(64, device=DEV)
    with pytest.raises(dsa.DSAError) as e:
        dsa.forward_static_ws(p, t, t, t, t, t, t, t, t, t)
    assert e.value.code == dsa.DSA_ERR_UNSUPPORTED
