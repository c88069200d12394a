"""Pins of the oracle's probe gate and kappa-gram check against closed forms,
exact rational arithmetic and brute force (no GPU)."""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def test_probe_closed_form_score():
    # h = alpha * w/|w|^2 + noise orthogonal to w  =>  w.h = alpha (before the cast)
    rng = np.random.default_rng(1)
    for d, h_dtype in [(64, "f32"), (4096, "bf16"), (8192, "bf16")]:
        alphas = np.array([-3.0, -0.5, 0.0, 0.4, 2.2])
        h, w = WL._probe_pair(rng, d, alphas, h_dtype)
        score, on, S = O.probe_gate(h, h_dtype, w, 0.4)
        # exact value of w.h for the stored (cast) h, from rationals
        hv = O.to_f64(h, h_dtype)
        for b in range(len(alphas)):
            exact = sum(Fraction(float(x)) * Fraction(float(y)) for x, y in zip(hv[b], w.astype(np.float64)))
            # fixed point sum differs from the exact sum by < d * 2^-32 (truncation per term)
            assert abs(Fraction(int(S[b]), 2 ** 32) - exact) < Fraction(d, 2 ** 32)
            # the cast moved w.h away from alpha by at most sum |dh_i w_i|
            assert abs(float(exact) - alphas[b]) < 0.05
            assert score[b] == pytest.approx(1 / (1 + math.exp(-float(exact))), abs=1e-6)
        assert list(on) == [False, False, True, True, True]  # logit(0.4) = -0.405


def test_probe_zero_vectors_give_one_half():
    w = _f32(np.random.default_rng(0).standard_normal(32))
    h = np.zeros((1, 32), dtype=np.float32)
    for hh, ww in [(h, w), (_f32(np.ones((1, 32))), np.zeros(32, np.float32))]:
        score, on, S = O.probe_gate(hh, "f32", ww, 0.4)
        assert S[0] == 0 and score[0] == 0.5 and on[0]
        score, on, S = O.probe_gate(hh, "f32", ww, 0.6)
        assert not on[0]


def test_probe_threshold_is_at_least_tau():
    # Build h, w whose fixed-point sum is exactly T (on) and T-1 (off):
    # sigma(s) >= tau  <=>  s >= logit(tau); "τ 이상" means at least tau.
    for tau in [0.4, 0.5, 0.1, 0.9, 0.73]:
        T = O.probe_threshold_fixed(tau)
        t32 = float(np.float32(tau))
        assert T == math.ceil(math.log(t32 / (1 - t32)) * 2 ** 32)
        for target, expect in [(T, True), (T - 1, False), (T + 1, True)]:
            hi = (target >> 20) << 20           # top bits, exact in fp32
            lo = target - hi                    # < 2^20, exact in fp32
            h = _f32([[hi * 2.0 ** -32, lo * 2.0 ** -32]])
            w = _f32([1.0, 1.0])
            score, on, S = O.probe_gate(h, "f32", w, tau)
            assert int(S[0]) == target
            assert bool(on[0]) == expect
            # and the decision agrees with the real-number definition sigma(s) >= tau
            s = target * 2.0 ** -32
            assert (1 / (1 + math.exp(-s)) >= t32) == expect or abs(s - math.log(t32 / (1 - t32))) < 1e-9


def test_probe_tau_limits():
    h = _f32([[100.0]]); w = _f32([1.0])
    assert O.probe_gate(h, "f32", w, 0.0)[1][0]
    assert not O.probe_gate(h, "f32", w, 1.0)[1][0]
    assert O.probe_gate(-h, "f32", w, -0.5)[1][0]


def test_probe_sum_order_independent():
    rng = np.random.default_rng(7)
    d = 4096
    h = WL.f32_to_bf16_bits(rng.standard_normal((3, d)).astype(np.float32))
    w = _f32(rng.standard_normal(d) / 64)
    S1 = O.probe_fixed_sum(h, "bf16", w)
    p = rng.permutation(d)
    S2 = O.probe_fixed_sum(h[:, p], "bf16", w[p])
    assert np.array_equal(S1, S2)


# --------------------------------------------------------------------------
# kappa-gram and retrieval: brute force over every short binary context
# --------------------------------------------------------------------------
def _brute_ends(seq, kappa):
    """Earlier occurrences of the final kappa-gram, by string search, latest first."""
    n = len(seq)
    if n < kappa + 1:
        return []
    s = "".join(map(str, seq))
    g = s[n - kappa:]
    ends = []
    stop = n - 1                    # an occurrence must end at or before n-2
    while True:
        i = s.rfind(g, 0, stop)     # searches s[0:stop]; occurrence fully inside
        if i < 0:
            break
        ends.append(i + kappa - 1)
        stop = i + kappa - 1        # next: ending strictly before this one
    return ends


def test_kgram_and_retrieval_brute_force():
    for n in range(1, 11):
        for bits in itertools.product([0, 1], repeat=n):
            row = np.array(bits, dtype=np.int32)
            for kappa in (1, 2, 3):
                ends = _brute_ends(bits, kappa)
                got = list(O.kgram_match_ends(row, n, kappa))
                assert got == ends, (bits, kappa)
                ctx = row[None, :]
                for W in (1, 2, 3):
                    for D in (1, 2, 4):
                        bt, bl, nc = O.retrieve(ctx, np.array([n]), np.array([1]), kappa, W, D,
                                                0, 0, np.zeros((1, 0), np.int32))
                        assert nc[0] == min(W, len(ends))
                        for k in range(W):
                            if k < len(ends):
                                j = ends[k]
                                L = min(D, n - 1 - j)
                                assert L >= 1
                                assert bl[0, k] == L
                                assert list(bt[0, k, :L]) == list(bits[j + 1:j + 1 + L])
                                assert all(bt[0, k, L:] == -1)
                            else:
                                assert bl[0, k] == 0 and all(bt[0, k] == -1)


def test_retrieval_hand_cases():
    # periodic run: overlapping occurrences count
    row = np.array([7, 7, 7, 7, 7, 7], dtype=np.int32)
    assert list(O.kgram_match_ends(row, 6, 2)) == [4, 3, 2, 1]
    # n <= kappa: nothing
    assert len(O.kgram_match_ends(row, 2, 2)) == 0
    # no match
    assert len(O.kgram_match_ends(np.arange(20, dtype=np.int32), 20, 3)) == 0
    # a match ending at n-2 gives a length-1 candidate
    row = np.array([7, 7, 7], dtype=np.int32)
    bt, bl, nc = O.retrieve(row[None], np.array([3]), np.array([1]), 1, 2, 4, 0, 0,
                            np.zeros((1, 0), np.int32))
    assert list(bl[0]) == [1, 2] and list(bt[0, 0, :1]) == [7] and nc[0] == 2
    # continuations truncated at the current token: len = min(D, n-1-j)
    row = np.array([1, 2, 1, 2, 1, 2], dtype=np.int32)
    bt, bl, nc = O.retrieve(row[None], np.array([6]), np.array([1]), 2, 4, 5, 0, 0,
                            np.zeros((1, 0), np.int32))
    assert list(bl[0]) == [2, 4, 0, 0] and nc[0] == 2
    assert list(bt[0, 0, :2]) == [1, 2] and list(bt[0, 1, :4]) == [1, 2, 1, 2]
    # gate off: no copy candidates; chain block per policy
    chain = np.array([[5, 6, 7]], dtype=np.int32)
    bt, bl, nc = O.retrieve(row[None], np.array([6]), np.array([0]), 2, 2, 4, 3, 1, chain)
    assert list(bl[0]) == [0, 0, 3] and nc[0] == 0 and list(bt[0, 2, :3]) == [5, 6, 7]
    bt, bl, nc = O.retrieve(row[None], np.array([6]), np.array([1]), 2, 2, 4, 3, 1, chain)
    assert list(bl[0]) == [2, 4, 0]
    bt, bl, nc = O.retrieve(row[None], np.array([6]), np.array([1]), 2, 2, 4, 3, 2, chain)
    assert list(bl[0]) == [2, 4, 3]


def test_gate_needs_both_probe_and_match():
    rng = np.random.default_rng(3)
    d = 64
    h, w = WL._probe_pair(rng, d, np.array([2.0, 2.0, -2.0, -2.0]), "f32")
    rep = np.array([1, 2, 3, 4, 5, 9, 1, 2, 3, 4, 5], dtype=np.int32)
    norep = np.arange(11, dtype=np.int32)
    ctx = np.stack([rep, norep, rep, norep])
    score, on, gate, last = O.gate_match(ctx, np.full(4, 11), h, "f32", w, 0.4, 5)
    assert list(on) == [True, True, False, False]
    assert list(last) == [4, -1, 4, -1]
    assert list(gate) == [1, 0, 0, 0]
