"""Device status word: a bounded wait that runs out, out-of-range indices.
Nothing here faults or hangs the GPU: the wait gives up after its budget and
the kernel returns normally."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import DEV, empty_outputs, lib, params

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    dsa = lib()
    assert dsa.get_status() == 0
    dsa.selftest_wait_timeout(2_000_000)  # 2 ms on an mbarrier nothing completes
    assert dsa.get_status() == dsa.DSA_ERR_TIMEOUT
    assert dsa.get_status() == 0          # read-and-clear
    x = torch.ones(4, device=DEV) * 2     # the context is still usable
    assert float(x.sum()) == 8.0


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_out_of_range_index_is_reported(dtype):
    dsa = lib()
    wl = dict(synth.TINY) if dtype == "fp32" else dict(synth.v32(64, "t"), topk=16)
    wl["S"] = 64
    wl["topk"] = 16
    x = synth.make_inputs(wl, device=DEV)
    p = params(dsa, wl)
    idx = torch.arange(16, dtype=torch.int32, device=DEV).repeat(1, 64, 1)
    idx[0, 5, 3] = 64      # == S_k: out of range
    idx[0, 6, 0] = -5      # below -1
    o = empty_outputs(wl, 64, torch.float32 if dtype == "fp32" else torch.bfloat16)
    dsa.sparse_attn_fwd(p, x["q"], x["kv"], idx, o["out"], o["m"], o["l"])
    torch.cuda.synchronize()
    assert dsa.get_status() == dsa.DSA_ERR_INDEX
    assert torch.isfinite(o["out"].float()).all()


def test_bad_row_position_is_reported():
    dsa = lib()
    wl = dict(synth.TINY)
    x = synth.make_inputs(wl, device=DEV)
    rows = torch.tensor([3, 256], dtype=torch.int32, device=DEV)  # 256 == S_k
    p = params(dsa, wl, S_q=2, q_row_index=rows)
    sc = torch.randn(2, 256, device=DEV)
    idx = torch.empty(2, wl["topk"], dtype=torch.int32, device=DEV)
    dsa.topk(p, sc, 0, 2, idx)
    torch.cuda.synchronize()
    assert dsa.get_status() == dsa.DSA_ERR_INDEX
    assert idx[1].eq(-1).all()
