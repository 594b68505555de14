"""C++ CPU oracle (``oracle/dsa_ref.cpp``) -- TEST INFRASTRUCTURE.

Same functions and return values as ``oracle.dsa_oracle`` (the numpy oracle),
computed by an independent C++ implementation: plain double-precision loops,
one query row per task on ``threads`` std::thread workers.  Only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / oracle legs use
it; the CUDA library never does.

``build()`` compiles ``libdsa_ref.so`` next to the source with the system C++
compiler (``__graft_entry__.build()`` calls it); importing this module does not
build anything, and calling a function without the library raises.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "dsa_ref.cpp")
LIB = os.path.join(_HERE, "libdsa_ref.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no C++ compiler found to build the C++ oracle")
    tmp = LIB + ".tmp"
    r = subprocess.run([cxx, "-O2", "-std=c++20", "-fPIC", "-shared", "-pthread", SRC, "-o", tmp],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("building the C++ oracle failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run oracle.cpp.build() first")
        lib = ctypes.CDLL(LIB)
        L, D, I = ctypes.c_longlong, ctypes.c_double, ctypes.c_int
        P = ctypes.c_void_p
        lib.dsa_ref_indexer_scores.argtypes = [L, L, L, L, L, P, P, P, P, P, I]
        lib.dsa_ref_topk.argtypes = [L, L, L, P, P, P, I]
        lib.dsa_ref_sparse_attn_fwd.argtypes = [L, L, L, L, L, L, L, P, P, P, D, P, P, P, I]
        lib.dsa_ref_sparse_attn_bwd.argtypes = [L, L, L, L, L, L, L, P, P, P, P, P, P, P, D, P, P, I]
        lib.dsa_ref_indexer_kl_loss.argtypes = [L, L, L, L, L, L, L, L, P, P, P, P, P, D, P, P, P, P,
                                                P, P, P, I]
        lib.dsa_ref_hardware_threads.restype = ctypes.c_int
        for f in ("dsa_ref_indexer_scores", "dsa_ref_topk", "dsa_ref_sparse_attn_fwd",
                  "dsa_ref_sparse_attn_bwd", "dsa_ref_indexer_kl_loss"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def hardware_threads() -> int:
    return int(_load().dsa_ref_hardware_threads())


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if x.dtype.is_floating_point:
            x = x.double()
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i(x, dt):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=dt)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return hardware_threads() if threads is None else int(threads)


def positions(B: int, S_q: int, q_row_offset: int = 0, q_row_index=None) -> np.ndarray:
    """Global position of each local query row, [B, S_q] int64: q_row_index[t]
    if given, else q_row_offset + t ([HP-CP] DSA CP: query rows of a shard)."""
    if q_row_index is not None:
        return _i(q_row_index, np.int64).reshape(B, S_q).copy()
    return np.broadcast_to(q_row_offset + np.arange(S_q, dtype=np.int64), (B, S_q)).copy()


def indexer_scores(q_I, k_I, w, pos, threads=None) -> np.ndarray:
    q_I, k_I, w = _f64(q_I), _f64(k_I), _f64(w)
    B, S_q, H_I, d_I = q_I.shape
    S_k = k_I.shape[1]
    pos = _i(pos, np.int64).reshape(B * S_q)
    out = np.empty((B, S_q, S_k))
    _load().dsa_ref_indexer_scores(B, S_q, S_k, H_I, d_I, _p(q_I), _p(k_I), _p(w), _p(pos), _p(out),
                                   _threads(threads))
    return out


def topk_select(scores, pos, k: int, threads=None) -> np.ndarray:
    """Scores are compared as doubles: fp32 inputs widen exactly and keep their
    order, so this is the fp32 comparison."""
    sc = _f64(scores)
    B, S_q, S_k = sc.shape
    pos = _i(pos, np.int64).reshape(B * S_q)
    out = np.empty((B, S_q, k), dtype=np.int32)
    _load().dsa_ref_topk(B * S_q, S_k, k, _p(sc), _p(pos), _p(out), _threads(threads))
    return out


def sparse_attn_fwd(q, kv, idx, scale: float, d_v: int, threads=None):
    q, kv = _f64(q), _f64(kv)
    idx = _i(idx, np.int32)
    B, S_q, H, d_qk = q.shape
    S_k, k = kv.shape[1], idx.shape[-1]
    O = np.empty((B, S_q, H, d_v))
    m = np.empty((B, S_q, H))
    l = np.empty((B, S_q, H))
    _load().dsa_ref_sparse_attn_fwd(B, S_q, S_k, H, d_qk, d_v, k, _p(q), _p(kv), _p(idx),
                                    float(scale), _p(O), _p(m), _p(l), _threads(threads))
    return O, m, l


def sparse_attn_bwd(q, kv, idx, O, dO, m, l, scale: float, d_v: int, threads=None):
    q, kv, O, dO, m, l = _f64(q), _f64(kv), _f64(O), _f64(dO), _f64(m), _f64(l)
    idx = _i(idx, np.int32)
    B, S_q, H, d_qk = q.shape
    S_k, k = kv.shape[1], idx.shape[-1]
    dq = np.empty_like(q)
    dkv = np.zeros_like(kv)
    _load().dsa_ref_sparse_attn_bwd(B, S_q, S_k, H, d_qk, d_v, k, _p(q), _p(kv), _p(idx), _p(O),
                                    _p(dO), _p(m), _p(l), float(scale), _p(dq), _p(dkv),
                                    _threads(threads))
    return dq, dkv


def indexer_kl_loss(q, kv, idx, m, l, scale: float, q_I, k_I, w, threads=None):
    q, kv, m, l = _f64(q), _f64(kv), _f64(m), _f64(l)
    q_I, k_I, w = _f64(q_I), _f64(k_I), _f64(w)
    idx = _i(idx, np.int32)
    B, S_q, H, d_qk = q.shape
    S_k, k = kv.shape[1], idx.shape[-1]
    H_I, d_I = q_I.shape[2], q_I.shape[3]
    loss_rows = np.empty(B * S_q)
    dq_I = np.empty_like(q_I)
    dk_I = np.zeros_like(k_I)
    dw = np.empty_like(w)
    _load().dsa_ref_indexer_kl_loss(B, S_q, S_k, H, d_qk, H_I, d_I, k, _p(q), _p(kv), _p(idx), _p(m),
                                    _p(l), float(scale), _p(q_I), _p(k_I), _p(w), _p(loss_rows),
                                    _p(dq_I), _p(dk_I), _p(dw), _threads(threads))
    loss = 0.0
    for v in loss_rows:          # tokens in order
        loss += float(v)
    return loss, dq_I, dk_I, dw


def dsa_forward(q_I, k_I, w, q, kv, k: int, scale: float, d_v: int, q_row_offset: int = 0,
                q_row_index=None, threads=None):
    """Indexer scores -> top-k -> sparse attention; returns (scores, idx, O, m, l)."""
    B, S_q = q.shape[:2]
    pos = positions(B, S_q, q_row_offset, q_row_index)
    scores = indexer_scores(q_I, k_I, w, pos, threads)
    idx = topk_select(scores, pos, k, threads)
    O, m, l = sparse_attn_fwd(q, kv, idx, scale, d_v, threads)
    return scores, idx, O, m, l
