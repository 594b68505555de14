"""dsa_forward_static_ws, the forward for callers that cannot allocate device
memory (custom-operator hosts that provide only input/output buffers, loops
that must not call cudaMalloc): it must give the same results as dsa_forward
with a caller-provided workspace, on two calls in a row (the fixed ring keeps
the previous call's contents)."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import BF16_MAXABS, DEV, bf16_close, empty_outputs, lib, np64, params

pytestmark = pytest.mark.gpu


def test_static_ring_forward_matches_workspace_forward():
    dsa = lib()
    wl = synth.WORKLOADS["dsv32_S4096"]
    S = wl["S"]
    x = synth.make_inputs(wl, device=DEV)
    p = params(dsa, wl)
    ref = empty_outputs(wl, S, torch.bfloat16)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) // 4, device=DEV)
    dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], ref["idx"], ref["out"], ref["m"],
                ref["l"], ws)
    torch.cuda.synchronize()
    assert dsa.get_status() == 0
    for call in range(2):
        o = empty_outputs(wl, S, torch.bfloat16)
        dsa.forward_static_ws(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], o["idx"], o["out"],
                              o["m"], o["l"])
        torch.cuda.synchronize()
        assert dsa.get_status() == 0
        assert torch.equal(o["idx"], ref["idx"]), call
        ok, ma, mr = bf16_close(np64(o["out"]), np64(ref["out"]))
        assert ok, (call, ma, mr)
        assert np.abs(np64(o["m"]) - np64(ref["m"])).max() < 1e-4
        assert (np.abs(np64(o["l"]) - np64(ref["l"])) / np64(ref["l"])).max() < 1e-4


def test_static_ring_rejects_oversized_key_length():
    dsa = lib()
    p = dsa.make_params(B=1, S_q=4, S_k=3_000_000, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                        topk=16, scale=0.1, dtype="bf16")
    t = torch.empty(64, device=DEV)
    with pytest.raises(dsa.DSAError) as e:
        dsa.forward_static_ws(p, t, t, t, t, t, t, t, t, t)
    assert e.value.code == dsa.DSA_ERR_UNSUPPORTED
