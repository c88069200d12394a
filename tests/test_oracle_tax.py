"""Pins of the speculation-tax counts (SwitchSD "무엇인가": a copy draft accepted for 0
tokens pays the verification for nothing), by hand-counted cases and a property."""
import numpy as np

from oracle import ssd_oracle as O


def test_hand_counted():
    gate = np.array([1, 1, 0, 1, 1], np.int32)
    n_cand = np.array([2, 0, 3, 1, 4], np.int32)
    W = 2
    # chain block at index 2 is ignored by the copy counts
    acc = np.array([[0, 0, 5], [0, 0, 0], [4, 4, 0], [3, 0, 0], [1, 6, 2]], np.int32)
    # attempts: seq 0 (taxed), seq 3 (run 3), seq 4 (run 6); seq 1 has no candidate, seq 2 gate off
    np.testing.assert_array_equal(O.copy_stats(gate, n_cand, acc, W), [3, 1, 9, 5])


def test_counts_add_up_over_random_batches():
    rng = np.random.default_rng(31)
    for _ in range(50):
        B, W = int(rng.integers(1, 40)), int(rng.integers(1, 5))
        gate = rng.integers(0, 2, B).astype(np.int32)
        n_cand = rng.integers(0, W + 1, B).astype(np.int32)
        acc = rng.integers(0, 4, (B, W + 1)).astype(np.int32)
        a, t, tok, n = O.copy_stats(gate, n_cand, acc, W)
        att = (gate != 0) & (n_cand > 0)
        assert a == att.sum() and n == B and 0 <= t <= a
        assert tok == acc[att, :W].max(axis=1).sum() if a else tok == 0
        assert t == (acc[att, :W].max(axis=1) == 0).sum() if a else t == 0
