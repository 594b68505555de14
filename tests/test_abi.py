"""The C-ABI library builds, loads without a GPU, and exports every entry
point include/dsa.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_long_gb300 as dsa
    return dsa


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_symbols()
    for n in ["dsa_indexer_scores", "dsa_topk", "dsa_sparse_attn_fwd", "dsa_sparse_attn_bwd",
              "dsa_forward", "dsa_indexer_kl_loss_bwd", "dsa_get_status", "dsa_workspace_size"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    dsa = _lib()
    raw = ctypes.CDLL(dsa.LIB_PATH)
    for n in declared_symbols():
        assert hasattr(raw, n), n
    assert dsa.version() == 100


def test_params_struct_layout_matches_header():
    dsa = _lib()
    # 4 int32, 9 int64, float + int32, int64, pointer, int64
    assert ctypes.sizeof(dsa.dsa_params) == 16 + 9 * 8 + 8 + 8 + 8 + 8


def test_host_validation_without_gpu():
    # argument errors are found on the host before any CUDA call
    dsa = _lib()
    p = dsa.make_params(B=1, S_q=8, S_k=8, H=2, d_qk=8, d_v=4, H_I=2, d_I=4, topk=4, scale=0.5,
                        dtype="fp32")
    assert dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) == 8 * 8 * 4
    bad = dsa.make_params(B=1, S_q=8, S_k=8, H=2, d_qk=8, d_v=16, H_I=2, d_I=4, topk=4, scale=0.5,
                          dtype="fp32")
    assert dsa.lib.dsa_sparse_attn_fwd(ctypes.byref(bad), 16, 16, 16, 16, 16, 16, None, None) == \
        dsa.DSA_ERR_INVALID_ARG
    uly = dsa.make_params(B=1, S_q=8, S_k=8, H=2, d_qk=8, d_v=4, H_I=2, d_I=4, topk=4, scale=0.5,
                          dtype="fp32", cp_mode="ulysses")
    assert dsa.lib.dsa_topk(ctypes.byref(uly), 16, 0, 1, 16, None) == dsa.DSA_ERR_UNSUPPORTED
    tnd = dsa.make_params(B=2, S_q=8, S_k=8, H=2, d_qk=8, d_v=4, H_I=2, d_I=4, topk=4, scale=0.5,
                          dtype="fp32", layout="TND")
    assert dsa.lib.dsa_topk(ctypes.byref(tnd), 16, 0, 1, 16, None) == dsa.DSA_ERR_INVALID_ARG
    off = dsa.make_params(B=1, S_q=8, S_k=8, H=2, d_qk=8, d_v=4, H_I=2, d_I=4, topk=4, scale=0.5,
                          dtype="fp32", q_row_offset=1)
    assert dsa.lib.dsa_topk(ctypes.byref(off), 16, 0, 1, 16, None) == dsa.DSA_ERR_INVALID_ARG
    assert dsa.lib.dsa_topk(ctypes.byref(p), 16, 0, 9, 16, None) == dsa.DSA_ERR_INVALID_ARG
    assert dsa.lib.dsa_topk(None, 16, 0, 1, 16, None) == dsa.DSA_ERR_INVALID_ARG
    bf = dsa.make_params(B=1, S_q=8, S_k=8, H=64, d_qk=576, d_v=512, H_I=64, d_I=128, topk=4,
                         scale=0.5, dtype="bf16")
    assert dsa.lib.dsa_sparse_attn_fwd(ctypes.byref(bf), 16, 16, 16, 16, 16, 16, None, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    # the FP8 indexer flag adds the E4M3 operands and scales to the forward's
    # workspace; the scratch-free forward runs the bf16 indexer only
    f8 = dsa.make_params(B=1, S_q=64, S_k=64, H=128, d_qk=576, d_v=512, H_I=64, d_I=128, topk=16,
                         scale=0.5, dtype="bf16", flags=2)
    plain = dsa.make_params(B=1, S_q=64, S_k=64, H=128, d_qk=576, d_v=512, H_I=64, d_I=128, topk=16,
                            scale=0.5, dtype="bf16")
    assert dsa.workspace_size(f8, dsa.DSA_CALL_FORWARD) >= \
        dsa.workspace_size(plain, dsa.DSA_CALL_FORWARD) + 64 * 64 * 128 + 64 * 128 + 64 * 64 * 4 + 64 * 4
    assert dsa.lib.dsa_forward_static_ws(ctypes.byref(f8), *([16] * 9), None) == dsa.DSA_ERR_UNSUPPORTED
    fp32 = dsa.make_params(B=1, S_q=8, S_k=8, H=2, d_qk=8, d_v=4, H_I=2, d_I=4, topk=4, scale=0.5,
                           dtype="fp32")
    assert dsa.lib.dsa_indexer_scores_fp8(ctypes.byref(fp32), 16, 16, 16, 16, 16, 0, 1, 16, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    # the bf16 path stores O with TMA: q, kv and out must be 16-byte aligned
    ds = dsa.make_params(B=1, S_q=8, S_k=8, H=128, d_qk=576, d_v=512, H_I=64, d_I=128, topk=4,
                         scale=0.5, dtype="bf16")
    assert dsa.lib.dsa_sparse_attn_fwd(ctypes.byref(ds), 16, 16, 16, 24, 16, 16, None, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert dsa.lib.dsa_sparse_attn_fwd(ctypes.byref(ds), 16, 8, 16, 16, 16, 16, None, None) == \
        dsa.DSA_ERR_INVALID_ARG


def test_backward_workspace_sizes():
    # bf16 tensor-core backward: P and scale*dS as bf16 hi/lo pairs
    # [rows*128][k] plus D [rows*128] fp32; the KL pass: head-summed P
    # [rows][k] fp32
    dsa = _lib()
    rows, k = 24, 2048
    p = dsa.make_params(B=1, S_q=rows, S_k=16384, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                        topk=k, scale=0.5, dtype="bf16")
    rh = rows * 128
    assert dsa.workspace_size(p, dsa.DSA_CALL_ATTN_BWD) == 4 * rh * k * 2 + rh * 4 + 256
    assert dsa.workspace_size(p, dsa.DSA_CALL_KL_BWD) == rows * k * 4 + 256
    # the fused backward: the attention backward's workspace, then the KL target
    assert dsa.workspace_size(p, dsa.DSA_CALL_BACKWARD) == \
        (4 * rh * k * 2 + rh * 4 + 256) + (rows * k * 4 + 256)
    # row passes (0 < wave_rows < S_q): the workspace holds one pass of
    # wave_rows rows whatever B and S_q are; wave_rows >= S_q is one pass
    for B, S_q, W in ((1, 24, 10), (3, 24, 10), (2, 100, 7)):
        pw = dsa.make_params(B=B, S_q=S_q, S_k=16384, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                             topk=k, scale=0.5, dtype="bf16", wave_rows=W)
        wh = W * 128
        assert dsa.workspace_size(pw, dsa.DSA_CALL_ATTN_BWD) == 4 * wh * k * 2 + wh * 4 + 256
        assert dsa.workspace_size(pw, dsa.DSA_CALL_KL_BWD) == W * k * 4 + 256
        assert dsa.workspace_size(pw, dsa.DSA_CALL_BACKWARD) == \
            (4 * wh * k * 2 + wh * 4 + 256) + (W * k * 4 + 256)
    whole = dsa.make_params(B=1, S_q=rows, S_k=16384, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                            topk=k, scale=0.5, dtype="bf16", wave_rows=rows)
    assert dsa.workspace_size(whole, dsa.DSA_CALL_ATTN_BWD) == dsa.workspace_size(p, dsa.DSA_CALL_ATTN_BWD)
    # a k that is not a multiple of 8 has no tensor-core backward
    odd = dsa.make_params(B=1, S_q=rows, S_k=16384, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                          topk=2047, scale=0.5, dtype="bf16")
    assert dsa.workspace_size(odd, dsa.DSA_CALL_ATTN_BWD) == 0
    assert dsa.lib.dsa_sparse_attn_bwd(ctypes.byref(odd), 16, 16, 16, 16, 16, 16, 16, 16, 16, 16,
                                       None) == dsa.DSA_ERR_UNSUPPORTED
    # the tensor-core backward needs its workspace
    assert dsa.lib.dsa_sparse_attn_bwd(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, 16, None,
                                       None) == dsa.DSA_ERR_WORKSPACE


def test_fused_indexer_topk_workspace_and_rejections():
    # dsa_indexer_topk (and dsa_forward with DSA_FLAG_FUSED_TOPK) keep one
    # wave's candidate lists: keys and positions (4 bytes each per key) and a
    # count per row; bf16 DeepSeek indexer shapes with S_k < 65536 only
    dsa = _lib()
    mk = lambda **kw: dsa.make_params(**dict(dict(B=1, S_q=64, S_k=64, H=128, d_qk=576, d_v=512,
                                                  H_I=64, d_I=128, topk=16, scale=0.5, dtype="bf16",
                                                  wave_rows=64), **kw))
    p = mk()
    W, S = 64, 64
    need = 2 * W * S * 4 + W * 4
    assert dsa.workspace_size(p, dsa.DSA_CALL_INDEXER_TOPK) >= need
    assert dsa.workspace_size(mk(flags=dsa.DSA_FLAG_FUSED_TOPK), dsa.DSA_CALL_FORWARD) >= need
    # the plain forward's ring is unchanged by the new call
    assert dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) == W * S * 4
    # unsupported: fp32, other indexer shapes, S_k >= 65536, with the FP8 flag
    for bad in (mk(dtype="fp32"), mk(H_I=32), mk(S_k=65536, S_q=64),
                mk(flags=dsa.DSA_FLAG_FUSED_TOPK | dsa.DSA_FLAG_FP8_INDEXER)):
        assert dsa.workspace_size(bad, dsa.DSA_CALL_INDEXER_TOPK) == 0
        assert dsa.lib.dsa_indexer_topk(ctypes.byref(bad), 16, 16, 16, 0, 1, 16, 16, None) == \
            dsa.DSA_ERR_UNSUPPORTED
    # argument checks happen on the host, before any launch
    assert dsa.lib.dsa_indexer_topk(ctypes.byref(p), 16, 16, 16, 0, 65, 16, 16, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert dsa.lib.dsa_indexer_topk(ctypes.byref(p), 16, 16, 16, 0, 1, 16, None, None) == \
        dsa.DSA_ERR_WORKSPACE
    assert dsa.lib.dsa_forward_static_ws(ctypes.byref(mk(flags=dsa.DSA_FLAG_FUSED_TOPK)),
                                         *([16] * 9), None) == dsa.DSA_ERR_UNSUPPORTED
