"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module holds no arithmetic of the attention method: it only turns
(seed, stream, element index) into pseudo-random numbers.

Generator (counter based, so any element can be produced independently and
every tensor is prefix-stable: the first rows of a long tensor equal the rows
of a shorter tensor drawn with the same seed and stream):

    G      = 0x9E3779B97F4A7C15                    (SplitMix64 increment)
    mix(z) = SplitMix64 finaliser:
             z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
             z ^= z >> 27; z *= 0x94D049BB133111EB
             z ^= z >> 31
    key    = mix(seed * G + stream)
    z1     = mix(key + (2 i + 1) * G),  z2 = mix(key + (2 i + 2) * G)
    u1     = ((z1 >> 11) + 1) * 2^-53   in (0, 1]
    u2     = (z2 >> 11) * 2^-53         in [0, 1)
    x_i    = sqrt(-2 ln u1) * cos(2 pi u2)      (Box-Muller, fp64)

all arithmetic mod 2^64.  The value is multiplied by ``scale`` in fp64 and then
rounded once to the requested dtype (torch's round-to-nearest-even).

Tensor stream ids (fixed ordinals): q_I=0, k_I=1, w=2, q=3, kv=4, dO=5.
"""
from __future__ import annotations

import math

import torch

STREAM = {"q_I": 0, "k_I": 1, "w": 2, "q": 3, "kv": 4, "dO": 5}

_G = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def _s64(u: int) -> int:
    """Unsigned 64-bit constant -> the int64 with the same bits."""
    u &= _MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def _srl(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = z ^ _srl(z, 30)
    z = z * _s64(_M1)
    z = z ^ _srl(z, 27)
    z = z * _s64(_M2)
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    z &= _MASK64
    z ^= z >> 30
    z = (z * _M1) & _MASK64
    z ^= z >> 27
    z = (z * _M2) & _MASK64
    return z ^ (z >> 31)


def normal_flat(start: int, count: int, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """fp64 standard normals for flat element indices [start, start+count)."""
    key = _mix_int(seed * _G + stream)
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    base = torch.full_like(i, _s64(key))
    c1 = base + (2 * i + 1) * _s64(_G)
    c2 = base + (2 * i + 2) * _s64(_G)
    z1 = _mix(c1)
    z2 = _mix(c2)
    u1 = (_srl(z1, 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = _srl(z2, 11).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal(shape, name_or_stream, seed: int = 0, scale: float = 1.0,
           dtype=torch.bfloat16, device="cpu", chunk: int = 1 << 24) -> torch.Tensor:
    """Tensor of N(0,1)*scale rounded to ``dtype``, generated on ``device``."""
    stream = STREAM[name_or_stream] if isinstance(name_or_stream, str) else int(name_or_stream)
    n = 1
    for d in shape:
        n *= int(d)
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        v = normal_flat(s, c, seed, stream, device=device)
        if scale != 1.0:
            v = v * scale
        out[s:s + c] = v.to(dtype)
    return out.view(*shape)


# --------------------------------------------------------------------------
# Workload recipes.  Shapes and distributions of the DeepSeek-V3.2 DSA
# configuration: 128 query heads, d_qk = 576 (512 latent + 64 rope), one
# shared kv row, d_v = 512, indexer 64 heads x 128, top-2048, softmax scale
# 1/sqrt(192); a tiny fp32 case for exact-arithmetic parity.
# --------------------------------------------------------------------------

TINY = dict(name="tiny_fp32_S256", B=1, S=256, H=8, d_qk=80, d_v=64, H_I=4, d_I=32,
            topk=32, scale=1.0 / math.sqrt(80.0), dtype="fp32")


def v32(S: int, name: str) -> dict:
    return dict(name=name, B=1, S=S, H=128, d_qk=576, d_v=512, H_I=64, d_I=128,
                topk=2048, scale=1.0 / math.sqrt(192.0), dtype="bf16")


WORKLOADS = {
    "tiny_fp32_S256": TINY,
    "dsv32_S4096": v32(4096, "dsv32_S4096"),
    "dsv32_S32768": v32(32768, "dsv32_S32768"),
    "dsv32_S16384_train": v32(16384, "dsv32_S16384_train"),
}


def head_tail_rows(S: int, cp: int, rank: int) -> torch.Tensor:
    """Global positions owned by ``rank`` under head-tail balancing: the
    sequence is cut into 2*cp chunks and rank r keeps chunks r and 2*cp-1-r."""
    assert S % (2 * cp) == 0
    c = S // (2 * cp)
    a = torch.arange(rank * c, (rank + 1) * c, dtype=torch.int32)
    b = torch.arange((2 * cp - 1 - rank) * c, (2 * cp - rank) * c, dtype=torch.int32)
    return torch.cat([a, b])


def make_inputs(wl: dict, device="cpu", seed: int = 0, with_dout: bool = False,
                S_q: int | None = None) -> dict:
    """All inputs of one workload.  fp32 workloads scale q_I, k_I by 1/sqrt(d_I)
    and q, kv by 1/sqrt(d_qk) (w unscaled); bf16 workloads use unit normals and
    w * 1/8.  ``S_q`` draws only the first S_q query rows (prefix-stable)."""
    B, S = wl["B"], wl["S"]
    Sq = S if S_q is None else S_q
    H, d_qk, d_v, H_I, d_I = wl["H"], wl["d_qk"], wl["d_v"], wl["H_I"], wl["d_I"]
    if wl["dtype"] == "fp32":
        dt = torch.float32
        sqi, ski, sw = 1.0 / math.sqrt(d_I), 1.0 / math.sqrt(d_I), 1.0
        sq, skv = 1.0 / math.sqrt(d_qk), 1.0 / math.sqrt(d_qk)
    else:
        dt = torch.bfloat16
        sqi = ski = sq = skv = 1.0
        sw = 1.0 / 8.0
    g = lambda shape, nm, sc: normal(shape, nm, seed, sc, dt, device)
    out = dict(
        q_I=g((B, Sq, H_I, d_I), "q_I", sqi),
        k_I=g((B, S, d_I), "k_I", ski),
        w=g((B, Sq, H_I), "w", sw),
        q=g((B, Sq, H, d_qk), "q", sq),
        kv=g((B, S, d_qk), "kv", skv),
    )
    if with_dout:
        out["dO"] = g((B, Sq, H, d_v), "dO", 1.0)
    return out
