"""Python binding of the GB300 DSA library (libdsa_gb300.so): argument
marshalling only.  Every step of the path runs in the library's CUDA kernels;
torch tensors are used for device memory and streams.

The library must be built first (``python -m sparse_attention_long_gb300._build``
or ``__graft_entry__.build()``); importing this module without it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_gb300.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE = 0, -1, -2, -3
DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_INDEX = -4, -5, -6
DSA_BSND, DSA_TND = 0, 1
DSA_BF16, DSA_FP32 = 0, 1
DSA_CP_COLOSSAL, DSA_CP_ULYSSES = 0, 1
DSA_CALL_FORWARD, DSA_CALL_ATTN_FWD, DSA_CALL_ATTN_BWD, DSA_CALL_KL_BWD, DSA_CALL_BACKWARD = 0, 1, 2, 3, 4
DSA_CALL_INDEXER_TOPK = 5
DSA_FLAG_CAUSAL_ONLY, DSA_FLAG_FP8_INDEXER, DSA_FLAG_FUSED_TOPK = 1, 2, 4

_ERRNAMES = {0: "DSA_OK", -1: "DSA_ERR_INVALID_ARG", -2: "DSA_ERR_UNSUPPORTED",
             -3: "DSA_ERR_WORKSPACE", -4: "DSA_ERR_CUDA", -5: "DSA_ERR_TIMEOUT", -6: "DSA_ERR_INDEX"}


class DSAError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {_ERRNAMES.get(code, code)}")
        self.code = code


class dsa_params(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("dtype", ctypes.c_int32), ("cp_mode", ctypes.c_int32),
                ("flags", ctypes.c_int32),
                ("B", ctypes.c_int64), ("S_q", ctypes.c_int64), ("S_k", ctypes.c_int64),
                ("H", ctypes.c_int64), ("d_qk", ctypes.c_int64), ("d_v", ctypes.c_int64),
                ("H_I", ctypes.c_int64), ("d_I", ctypes.c_int64), ("topk", ctypes.c_int64),
                ("scale", ctypes.c_float), ("reserved1", ctypes.c_int32),
                ("q_row_offset", ctypes.c_int64), ("q_row_index", ctypes.c_void_p),
                ("wave_rows", ctypes.c_int64)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                      "(nvcc, sm_103a); there is no fallback implementation")
lib = ctypes.CDLL(LIB_PATH)

_vp, _i64, _i32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p
_P = ctypes.POINTER(dsa_params)
_sigs = {
    "dsa_version": ([], ctypes.c_int),
    "dsa_workspace_size": ([_P, ctypes.c_int], ctypes.c_size_t),
    "dsa_indexer_scores": ([_P, _vp, _vp, _vp, _i64, _i64, _vp, _vp], ctypes.c_int),
    "dsa_indexer_quantize_fp8": ([_P] + [_vp] * 7, ctypes.c_int),
    "dsa_indexer_scores_fp8": ([_P, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp], ctypes.c_int),
    "dsa_topk": ([_P, _vp, _i64, _i64, _vp, _vp], ctypes.c_int),
    "dsa_indexer_topk": ([_P, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp], ctypes.c_int),
    "dsa_sparse_attn_fwd": ([_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "dsa_sparse_attn_bwd": ([_P] + [_vp] * 11, ctypes.c_int),
    "dsa_indexer_kl_loss_bwd": ([_P] + [_vp] * 14, ctypes.c_int),
    "dsa_backward": ([_P] + [_vp] * 18, ctypes.c_int),
    "dsa_forward": ([_P] + [_vp] * 11, ctypes.c_int),
    "dsa_forward_static_ws": ([_P] + [_vp] * 10, ctypes.c_int),
    "dsa_get_status": ([_vp, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "dsa_set_wait_budget_ns": ([ctypes.c_uint64], ctypes.c_int),
    "dsa_selftest_wait_timeout": ([ctypes.c_uint64, _vp], ctypes.c_int),
}
for _n, (_a, _r) in _sigs.items():
    _f = getattr(lib, _n)
    _f.argtypes, _f.restype = _a, _r


def _chk(rc: int, where: str):
    if rc != DSA_OK:
        raise DSAError(rc, where)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_params(*, B, S_q, S_k, H, d_qk, d_v, H_I, d_I, topk, scale, dtype="bf16",
                layout="BSND", q_row_offset=0, q_row_index=None, wave_rows=0,
                cp_mode="colossal", flags=0) -> dsa_params:
    """Builds the C parameter block.  ``q_row_index`` is a device int32 tensor
    (kept alive by the caller) or None."""
    p = dsa_params()
    p.layout = {"BSND": DSA_BSND, "TND": DSA_TND}[layout]
    p.dtype = {"bf16": DSA_BF16, "fp32": DSA_FP32}[dtype]
    p.cp_mode = {"colossal": DSA_CP_COLOSSAL, "ulysses": DSA_CP_ULYSSES}[cp_mode]
    p.B, p.S_q, p.S_k, p.H, p.d_qk, p.d_v = B, S_q, S_k, H, d_qk, d_v
    p.H_I, p.d_I, p.topk, p.scale = H_I, d_I, topk, float(scale)
    p.q_row_offset = q_row_offset
    p.q_row_index = None if q_row_index is None else _ptr(q_row_index)
    p.wave_rows = wave_rows
    p.flags = flags
    return p


def wave_rows(p: dsa_params) -> int:
    """Rows per indexer/top-k wave dsa_forward uses: its plain score ring holds
    one wave of S_k fp32 scores per row, so the library's workspace size for
    the same shape without the indexer flags gives it."""
    q = dsa_params.from_buffer_copy(p)
    q.flags &= ~(DSA_FLAG_FP8_INDEXER | DSA_FLAG_FUSED_TOPK)
    return workspace_size(q, DSA_CALL_FORWARD) // (4 * q.S_k)


def version() -> int:
    return lib.dsa_version()


def workspace_size(p: dsa_params, which: int) -> int:
    return lib.dsa_workspace_size(ctypes.byref(p), which)


def indexer_scores(p, q_I, k_I, w, row_begin, rows, scores, stream=None):
    _chk(lib.dsa_indexer_scores(ctypes.byref(p), _ptr(q_I), _ptr(k_I), _ptr(w), row_begin, rows,
                                _ptr(scores), _stream(stream)), "dsa_indexer_scores")


def indexer_quantize_fp8(p, q_I, k_I, q8, q_scale, k8, k_scale, stream=None):
    _chk(lib.dsa_indexer_quantize_fp8(ctypes.byref(p), _ptr(q_I), _ptr(k_I), _ptr(q8), _ptr(q_scale),
                                      _ptr(k8), _ptr(k_scale), _stream(stream)),
         "dsa_indexer_quantize_fp8")


def indexer_scores_fp8(p, q8, q_scale, k8, k_scale, w, row_begin, rows, scores, stream=None):
    _chk(lib.dsa_indexer_scores_fp8(ctypes.byref(p), _ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale),
                                    _ptr(w), row_begin, rows, _ptr(scores), _stream(stream)),
         "dsa_indexer_scores_fp8")


def topk(p, scores, row_begin, rows, idx, stream=None):
    _chk(lib.dsa_topk(ctypes.byref(p), _ptr(scores), row_begin, rows, _ptr(idx), _stream(stream)),
         "dsa_topk")


def indexer_topk(p, q_I, k_I, w, row_begin, rows, idx, workspace, stream=None):
    """Fused indexer + streaming top-k: the indices dsa_indexer_scores +
    dsa_topk give, without a score matrix (workspace: DSA_CALL_INDEXER_TOPK)."""
    _chk(lib.dsa_indexer_topk(ctypes.byref(p), _ptr(q_I), _ptr(k_I), _ptr(w), row_begin, rows,
                              _ptr(idx), _ptr(workspace), _stream(stream)), "dsa_indexer_topk")


def sparse_attn_fwd(p, q, kv, idx, out, softmax_max, softmax_sum, workspace=None, stream=None):
    _chk(lib.dsa_sparse_attn_fwd(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(out),
                                 _ptr(softmax_max), _ptr(softmax_sum), _ptr(workspace),
                                 _stream(stream)), "dsa_sparse_attn_fwd")


def sparse_attn_bwd(p, q, kv, idx, out, dout, softmax_max, softmax_sum, dq, dkv, workspace=None,
                    stream=None):
    _chk(lib.dsa_sparse_attn_bwd(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(out),
                                 _ptr(dout), _ptr(softmax_max), _ptr(softmax_sum), _ptr(dq),
                                 _ptr(dkv), _ptr(workspace), _stream(stream)), "dsa_sparse_attn_bwd")


def indexer_kl_loss_bwd(p, q, kv, q_I, k_I, w, idx, softmax_max, softmax_sum, loss, dq_I, dk_I, dw,
                        workspace=None, stream=None):
    _chk(lib.dsa_indexer_kl_loss_bwd(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(q_I), _ptr(k_I),
                                     _ptr(w), _ptr(idx), _ptr(softmax_max), _ptr(softmax_sum),
                                     _ptr(loss), _ptr(dq_I), _ptr(dk_I), _ptr(dw),
                                     _ptr(workspace), _stream(stream)), "dsa_indexer_kl_loss_bwd")


def backward(p, q, kv, idx, out, dout, softmax_max, softmax_sum, q_I, k_I, w, dq, dkv, loss, dq_I,
             dk_I, dw, workspace=None, stream=None):
    """sparse_attn_bwd and indexer_kl_loss_bwd in one call sharing the recompute of P."""
    _chk(lib.dsa_backward(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(out), _ptr(dout),
                          _ptr(softmax_max), _ptr(softmax_sum), _ptr(q_I), _ptr(k_I), _ptr(w),
                          _ptr(dq), _ptr(dkv), _ptr(loss), _ptr(dq_I), _ptr(dk_I), _ptr(dw),
                          _ptr(workspace), _stream(stream)), "dsa_backward")


def forward(p, q_I, k_I, w, q, kv, idx_out, out, softmax_max, softmax_sum, workspace, stream=None):
    _chk(lib.dsa_forward(ctypes.byref(p), _ptr(q_I), _ptr(k_I), _ptr(w), _ptr(q), _ptr(kv),
                         _ptr(idx_out), _ptr(out), _ptr(softmax_max), _ptr(softmax_sum),
                         _ptr(workspace), _stream(stream)), "dsa_forward")


def forward_static_ws(p, q_I, k_I, w, q, kv, idx_out, out, softmax_max, softmax_sum, stream=None):
    """dsa_forward without a workspace argument: the score ring is the
    library's own fixed device array (for callers that cannot allocate)."""
    _chk(lib.dsa_forward_static_ws(ctypes.byref(p), _ptr(q_I), _ptr(k_I), _ptr(w), _ptr(q),
                                   _ptr(kv), _ptr(idx_out), _ptr(out), _ptr(softmax_max),
                                   _ptr(softmax_sum), _stream(stream)), "dsa_forward_static_ws")


def get_status(stream=None) -> int:
    v = ctypes.c_int(0)
    _chk(lib.dsa_get_status(_stream(stream), ctypes.byref(v)), "dsa_get_status")
    return v.value


def set_wait_budget_ns(ns: int):
    _chk(lib.dsa_set_wait_budget_ns(int(ns)), "dsa_set_wait_budget_ns")


def selftest_wait_timeout(ns: int, stream=None):
    _chk(lib.dsa_selftest_wait_timeout(int(ns), _stream(stream)), "dsa_selftest_wait_timeout")
