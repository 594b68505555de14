"""The seeded input generator: published SplitMix64 vector, determinism,
prefix stability, and rough N(0,1) moments."""
import torch

import synth


def test_splitmix64_reference_vector():
    # Vigna's SplitMix64 reference outputs for state 1234567.
    G = 0x9E3779B97F4A7C15
    got = [synth._mix_int(1234567 + j * G) for j in range(1, 6)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]
    z = synth._mix(torch.tensor([synth._s64(1234567 + j * G) for j in range(1, 6)], dtype=torch.int64))
    assert [int(v) & ((1 << 64) - 1) for v in z] == got


def test_prefix_stable_and_deterministic():
    a = synth.normal((64, 3, 5), "q", 0, 1.0, torch.float32)
    b = synth.normal((16, 3, 5), "q", 0, 1.0, torch.float32)
    assert torch.equal(a[:16], b)
    assert torch.equal(a, synth.normal((64, 3, 5), "q", 0, 1.0, torch.float32))
    assert not torch.equal(a, synth.normal((64, 3, 5), "kv", 0, 1.0, torch.float32))


def test_moments():
    x = synth.normal((1 << 18,), "kv", 0, 1.0, torch.float64)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
