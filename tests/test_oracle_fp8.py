"""Pins for the FP8 (E4M3) indexer oracle (oracle/fp8.py, CPU only).

E4M3 rounding is pinned by hand-worked values (ties, saturation, subnormals),
by every one of the 254 finite codes decoded from the bit layout, by the
midpoints between neighbouring codes, and by torch's float8_e4m3fn cast on
in-range values; the quantized indexer reduces to the bf16 oracle's formula
when the inputs are already E4M3 values with absmax 448 (scale 1)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def _decode(code: int) -> float:
    """Value of an E4M3 code from its bit layout: sign | 4-bit exponent (bias 7) | 3-bit mantissa."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]   # 0x7F / 0xFF are NaN


def test_hand_values():
    cases = [
        (1.0, 1.0), (1.0625, 1.0),          # tie between 1 and 1.125: even mantissa
        (1.1875, 1.25),                     # tie between 1.125 and 1.25: even (mantissa 2)
        (448.0, 448.0), (464.0, 448.0),     # tie between 448 and the NaN slot: even, 448
        (470.0, 448.0), (1e6, 448.0),       # saturate
        (2.0 ** -9, 2.0 ** -9),             # smallest subnormal
        (2.0 ** -10, 0.0),                  # tie between 0 and 2^-9: even, 0
        (3 * 2.0 ** -10, 2.0 ** -8),        # tie between 2^-9 and 2^-8: even
        (0.0, 0.0), (-3.3, -3.25), (0.017, 0.017578125),
    ]
    for x, want in cases:
        assert fp8.e4m3_round(np.float64(x)) == want, (x, want)


def test_every_finite_code_is_a_fixed_point():
    vals = np.array([_decode(c) for c in FINITE])
    assert vals.max() == 448.0 and vals.min() == -448.0
    np.testing.assert_array_equal(fp8.e4m3_round(vals), vals)


def test_midpoints_round_to_the_even_neighbour():
    pos = sorted({_decode(c) for c in FINITE if _decode(c) >= 0})
    for a, b in zip(pos[:-1], pos[1:]):
        mid = (a + b) / 2.0
        # the neighbour with an even mantissa (its code's lowest bit is 0)
        codes = {_decode(c): c for c in FINITE if _decode(c) >= 0}
        want = a if codes[a] % 2 == 0 else b
        assert fp8.e4m3_round(mid) == want, (a, b)
        assert fp8.e4m3_round(np.nextafter(mid, 0.0)) == a
        assert fp8.e4m3_round(np.nextafter(mid, 1e9)) == b


def test_matches_torch_float8_cast_in_range():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, size=20000))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x), ref)


def test_quantize_rows():
    v = np.array([[0.5, -2.0, 0.25, 1.0], [0.0, 0.0, 0.0, 0.0]], dtype=np.float32)
    q, s = fp8.quantize_rows(v)
    assert s[0] == np.float32(2.0) / np.float32(448.0) and s[1] == 1.0
    assert q[0, 1] == -448.0                        # the absmax element hits the top code
    assert np.all(q[1] == 0.0)
    # every element dequantizes to within half an E4M3 quantum of its value
    deq = q[0] * s[0]
    assert np.all(np.abs(deq - v[0]) <= np.abs(v[0]) * 2.0 ** -4 + 1e-12)


def test_reduces_to_the_bf16_formula_on_e4m3_inputs():
    # inputs that are E4M3 values with absmax 448 in every vector: scale 1,
    # quantization is the identity, scores equal the unquantized oracle's
    rng = np.random.default_rng(5)
    codes = np.array([_decode(c) for c in FINITE])
    B, S, H, d = 1, 9, 3, 128
    qI = rng.choice(codes, size=(B, S, H, d))
    kI = rng.choice(codes, size=(B, S, d))
    qI[..., 0] = 448.0
    kI[..., 0] = -448.0
    w = rng.standard_normal((B, S, H))
    pos = oracle.positions(B, S)
    np.testing.assert_array_equal(fp8.indexer_scores_fp8(qI, kI, w, pos),
                                  oracle.indexer_scores(qI, kI, w, pos))


def test_quantization_error_is_bounded():
    # each element moves by at most half an E4M3 quantum: 2^-4 |x| in the
    # normal range, 2^-10 * scale among the subnormals; the score then moves by
    # at most sum_j w_j sum_d (e_q |k| + |q| e_k + e_q e_k) -- a property of
    # any correct quantizer, independent of how this one is written
    rng = np.random.default_rng(9)
    B, S, H, d = 1, 17, 4, 128
    qI = rng.standard_normal((B, S, H, d)).astype(np.float32)
    kI = rng.standard_normal((B, S, d)).astype(np.float32)
    w = np.abs(rng.standard_normal((B, S, H)))
    pos = oracle.positions(B, S)
    a = fp8.indexer_scores_fp8(qI, kI, w, pos)
    b = oracle.indexer_scores(qI, kI, w, pos)
    fin = np.isfinite(b)
    sq = np.abs(qI).max(-1, keepdims=True) / 448.0
    sk = np.abs(kI).max(-1, keepdims=True) / 448.0
    eq = np.maximum(2.0 ** -4 * np.abs(qI), 2.0 ** -10 * sq) * (1 + 1e-6)
    ek = np.maximum(2.0 ** -4 * np.abs(kI), 2.0 ** -10 * sk) * (1 + 1e-6)
    Q, K, EQ, EK = (np.asarray(v, np.float64) for v in (qI, kI, eq, ek))
    term = (EQ[:, :, :, None, :] * np.abs(K)[:, None, None, :, :] + np.abs(Q)[:, :, :, None, :] * EK[:, None, None, :, :]
            + EQ[:, :, :, None, :] * EK[:, None, None, :, :]).sum(-1)
    bound = (w[..., None] * term).sum(2)
    assert np.all(np.abs(a[fin] - b[fin]) <= bound[fin] + 1e-12)
