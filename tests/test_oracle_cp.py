"""Pins for the CP-shard row mapping (CPU only): a shard's rows equal the same
rows of the unsharded run, for offsets and for head-tail row lists."""
import numpy as np
import torch

import synth
from oracle import dsa_forward, positions


def _inputs(S, seed=3):
    rng = np.random.default_rng(seed)
    H_I, d_I, H, d_qk = 2, 8, 3, 12
    return dict(q_I=rng.standard_normal((1, S, H_I, d_I)), k_I=rng.standard_normal((1, S, d_I)),
                w=rng.standard_normal((1, S, H_I)), q=rng.standard_normal((1, S, H, d_qk)),
                kv=rng.standard_normal((1, S, d_qk)))


def test_head_tail_rows():
    r = synth.head_tail_rows(32, 4, 1).tolist()
    assert r == [4, 5, 6, 7, 24, 25, 26, 27]
    allr = sorted(sum((synth.head_tail_rows(32, 4, k).tolist() for k in range(4)), []))
    assert allr == list(range(32))


def test_positions():
    assert positions(1, 3, 5).tolist() == [[5, 6, 7]]
    assert positions(2, 2, 0, np.array([3, 9, 1, 2])).tolist() == [[3, 9], [1, 2]]


def _run(x, k, rows=None, off=0, ridx=None):
    pick = (lambda a: a) if rows is None else (lambda a: a[:, rows])
    return dsa_forward(pick(x["q_I"]), x["k_I"], pick(x["w"]), pick(x["q"]), x["kv"], k, 0.4, 8,
                       q_row_offset=off, q_row_index=ridx)


def test_offset_shard_rows_identical():
    S, k = 48, 6
    x = _inputs(S)
    full = _run(x, k)
    rows = np.arange(20, 30)
    part = _run(x, k, rows=rows, off=20)
    for a, b in zip(part, full):
        np.testing.assert_array_equal(a, b[:, rows])


def test_head_tail_shard_rows_identical():
    S, k, cp = 48, 6, 4
    x = _inputs(S, seed=4)
    full = _run(x, k)
    for r in range(cp):
        rows = synth.head_tail_rows(S, cp, r).numpy()
        part = _run(x, k, rows=rows, ridx=rows)
        for a, b in zip(part, full):
            np.testing.assert_array_equal(a, b[:, rows])
