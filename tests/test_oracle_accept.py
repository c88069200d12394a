"""Pins of the oracle's vocabulary rows, acceptance and final draw against the
pages' worked cases, closed forms, exact counting and a chi-square test of
losslessness (no GPU)."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import ssd_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _accept_one(p_rows, q_rows, toks, u_acc, u_fin, chain=True, mode="sample"):
    """Run the oracle acceptance on one sequence with a single block given as
    probability rows: p_rows [L+1][V] (row d predicts token d+1), q_rows [L][V]."""
    L = len(toks)
    V = len(p_rows[0])
    tgt = np.zeros((1, 1 + L, V), np.float32)
    tgt[0, :] = np.asarray(p_rows, np.float32)
    blk_tok = np.asarray(toks, np.int32).reshape(1, 1, L)
    blk_len = np.array([[L]], np.int32)
    drf = np.asarray(q_rows, np.float32).reshape(1, L, V) if chain else None
    r = O.verify_step_accept(mode, "probs_f32", tgt, drf, blk_tok, blk_len, 0 if chain else 1,
                             1 if chain else 0, np.asarray(u_acc, np.float32).reshape(1, 1, L),
                             np.asarray([u_fin], np.float32))
    return r


# ---- a6 ---------------------------------------------------------------------
def test_softmax_rows_against_library_and_normalised():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((5, 1000)) * math.sqrt(3)).astype(np.float32)
    p64 = O.softmax_f64(x)
    np.testing.assert_allclose(p64.sum(axis=1), 1.0, atol=1e-12)
    np.testing.assert_allclose(p64, scipy.special.softmax(x.astype(np.float64), axis=1), rtol=1e-12)
    p32 = O.row_probs(x, "logits_f32")
    assert p32.dtype == np.float32
    np.testing.assert_allclose(p32, p64, rtol=2 ** -24)


def test_argmax_lowest_index_on_ties():
    x = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]], np.float32)
    assert list(O.first_argmax(x)) == [1, 0]


# ---- a7: the page's worked cases (SD-anatomy §5) ----------------------------
def test_case1_p_at_least_q_always_accepts():
    for u in [0.01, 0.5, 0.9999]:
        assert O.accept_test(u, 0.3, 0.7)
        assert O.accept_test(u, 0.4, 0.4)


def test_case2_threshold_at_p_over_q():
    # p/q = 0.5: u just below accepts, u at the ratio rejects (u*q < p is strict)
    assert O.accept_test(0.49, 0.6, 0.3)
    assert not O.accept_test(0.5, 0.6, 0.3)
    assert not O.accept_test(0.51, 0.6, 0.3)


def test_case3_residual_normalises_and_vanishes_where_q_exceeds_p():
    rng = np.random.default_rng(2)
    p = rng.dirichlet(np.ones(50)).astype(np.float32)
    q = rng.dirichlet(np.ones(50)).astype(np.float32)
    P, Q = O.prob_weights(p), O.prob_weights(q)
    R = O.residual_weights(P, Q)
    assert np.all(R[Q >= P] == 0) and np.all(R[P > Q] > 0)
    pr = R / R.sum()
    assert abs(pr.sum() - 1.0) < 1e-12
    # lossless identity (§3.3) holds exactly in integer weights: min(P,Q) + max(0,P-Q) = P
    assert np.array_equal(np.minimum(P, Q) + R, P)


def test_case4_bonus_token_golden():
    g = json.load(open(os.path.join(GOLDEN, "bonus_token_case.json")))
    voc = g["vocab"]
    toks = [voc.index(t) for t in g["draft_tokens"]]
    r = _accept_one(g["p_rows"], g["q_rows"], toks, g["u_acc"], g["u_fin"])
    assert r["n_out"][0] == 4
    assert [voc[i] for i in r["out_tok"][0, :4]] == g["expected_tokens"]
    assert r["acc_len"][0, 0] == 3


def test_q_equal_p_accepts_everything():
    rng = np.random.default_rng(4)
    V, L = 30, 6
    p = rng.dirichlet(np.ones(V), size=L + 1).astype(np.float32)
    toks = [int(rng.integers(V)) for _ in range(L)]
    u = rng.random(L).astype(np.float32) * np.float32(0.9999)
    r = _accept_one(p, p[:L], toks, u, 0.3)
    assert r["acc_len"][0, 0] == L and r["n_out"][0] == L + 1


def test_greedy_one_hot_gives_lcp_and_target_sequence():
    # one-hot target rows: the emitted tokens are exactly what the target alone
    # emits greedily (SD-lossless, 2단계), and the accepted length is the LCP
    rng = np.random.default_rng(5)
    V = 12
    for trial in range(50):
        L = int(rng.integers(1, 8))
        truth = rng.integers(0, V, size=L + 1)
        rows = np.eye(V, dtype=np.float32)[truth]               # row d predicts truth[d]
        toks = truth[:L].copy()
        cut = int(rng.integers(0, L + 1))
        if cut < L:
            toks[cut] = (truth[cut] + 1 + int(rng.integers(V - 1))) % V
        lcp = next((i for i in range(L) if toks[i] != truth[i]), L)
        for mode in ("greedy", "sample"):
            r = _accept_one(rows, rows[:L], toks, rng.random(L) * 0.999, float(rng.random()),
                            chain=False, mode=mode)
            assert r["acc_len"][0, 0] == lcp
            assert list(r["out_tok"][0, :lcp + 1]) == list(truth[:lcp + 1])


# ---- a8: the integer inverse CDF -----------------------------------------------
def test_draw_index_exact_counts_over_all_uniforms():
    rng = np.random.default_rng(6)
    Wt = rng.integers(0, 1 << 36, size=9).astype(np.int64)
    Wt[3] = 0
    S = int(Wt.sum())
    # every representable uniform k*2^-24: the count mapped to token i is within
    # one of W_i * 2^24 / S, tokens of zero weight are never drawn
    T = np.array([(int(u) * S) >> 24 for u in range(0, 1 << 24, 4096)], dtype=np.int64)
    C = np.cumsum(Wt)
    idx = np.searchsorted(C, T, side="right")
    assert 3 not in set(idx.tolist())
    counts = np.bincount(idx, minlength=9) * 4096
    expect = Wt / S * (1 << 24)
    assert np.all(np.abs(counts - expect) <= 4096 + 1)
    # and draw_index agrees with the direct definition on sampled uniforms
    for k in rng.integers(0, 1 << 24, size=200):
        u = float(k) * 2.0 ** -24
        Tt = (int(k) * S) >> 24
        direct = next(i for i in range(9) if int(C[i]) > Tt)
        assert O.draw_index(Wt, u) == direct


def test_selection_longest_then_lowest_block():
    V = 8
    Dmax = 3
    NB = 3
    eye = np.eye(V, dtype=np.float32)
    # block tokens; the target prefers token 1 everywhere
    tgt = np.tile(eye[1], (1, 1 + NB * Dmax, 1))
    blk_tok = np.array([[[1, 2, 2], [1, 1, 2], [1, 1, 5]]], np.int32)
    blk_len = np.array([[3, 3, 3]], np.int32)
    r = O.verify_step_accept("greedy", "probs_f32", tgt, None, blk_tok, blk_len, NB, 0,
                             np.zeros((1, NB, Dmax), np.float32), np.zeros(1, np.float32))
    assert list(r["acc_len"][0]) == [1, 2, 2]
    assert r["best_blk"][0] == 1 and r["n_out"][0] == 3
    assert list(r["out_tok"][0, :3]) == [1, 1, 1]
    # no block at all: one token from row 0
    r = O.verify_step_accept("greedy", "probs_f32", tgt, None, blk_tok, np.zeros((1, NB), np.int32), NB, 0,
                             np.zeros((1, NB, Dmax), np.float32), np.zeros(1, np.float32))
    assert r["best_blk"][0] == -1 and r["n_out"][0] == 1 and r["out_tok"][0, 0] == 1


def test_copy_residual_excludes_rejected_candidate():
    # one-hot q on the candidate: after a rejection the draw comes from p without x
    p = np.array([0.5, 0.3, 0.2], np.float32)
    rows = np.stack([p, p])
    for uf in np.linspace(0, 0.999, 37):
        r = _accept_one(rows, None, [0], [0.9], float(uf), chain=False)
        assert r["acc_len"][0, 0] == 0
        assert r["out_tok"][0, 0] in (1, 2)


# ---- lossless distribution (SD-anatomy §3.3, §5 Case 5) -----------------------
@pytest.mark.parametrize("V", [16, 64])
def test_chi_square_first_token_distribution_equals_p(V):
    rng = np.random.default_rng(100 + V)
    p = rng.dirichlet(np.ones(V) * 0.7).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.7).astype(np.float32)      # far from p
    N = 1_000_000
    B = N
    x = rng.choice(V, size=B, p=q.astype(np.float64) / q.sum())
    tgt = np.broadcast_to(np.stack([p, p])[None], (B, 2, V))
    drf = np.broadcast_to(q[None, None], (B, 1, V))
    u_acc = (rng.integers(0, 1 << 24, size=(B, 1, 1)) * 2.0 ** -24).astype(np.float32)
    u_fin = (rng.integers(0, 1 << 24, size=B) * 2.0 ** -24).astype(np.float32)
    counts = np.zeros(V, np.int64)
    # one chain block of length 1 per trial; batches keep memory small
    step = 100_000
    for s in range(0, B, step):
        sl = slice(s, s + step)
        r = O.verify_step_accept("sample", "probs_f32", tgt[sl], drf[sl], x[sl].reshape(-1, 1, 1).astype(np.int32),
                                 np.ones((step, 1), np.int32), 0, 2, u_acc[sl], u_fin[sl])
        counts += np.bincount(r["out_tok"][:, 0], minlength=V)
    expected = p.astype(np.float64) / p.sum() * N
    chi2, pval = scipy.stats.chisquare(counts, expected)
    assert pval > 0.01, (chi2, pval)


# ---- several copy blocks: the choice of the longest (sample mode) ---------------
def _two_block_categories(p, p1row, p2row, x1, x2):
    """Joint law of (chosen block, tokens emitted) for two one-token copy blocks with
    candidates x1 (block 0) and x2 (block 1), derived by hand from the rules: block k
    accepts with probability p(x_k) (one-hot q); the longer run wins, ties go to block 0;
    an accepted block adds a bonus token from the row after its token; when both reject,
    block 0 is chosen and its residual is p without x1."""
    V = len(p)
    pa, pb = float(p[x1]), float(p[x2])
    cats = {}
    for y in range(V):
        cats[(0, 2, x1, y)] = pa * float(p1row[y])
        cats[(1, 2, x2, y)] = (1.0 - pa) * pb * float(p2row[y])
        if y != x1:
            cats[(0, 1, y, -1)] = (1.0 - pb) * float(p[y])
    return cats


def test_two_copy_blocks_follow_their_closed_form_and_are_not_lossless():
    """Pins the selection across blocks in sample mode (the pages make no losslessness
    claim for it): longest run, lowest block on ties, residual of the chosen block."""
    rng = np.random.default_rng(2024)
    V, x1, x2 = 6, 1, 4
    p, p1row, p2row = (rng.dirichlet(np.full(V, 2.0)).astype(np.float32) for _ in range(3))
    N = 200_000
    tgt = np.broadcast_to(np.stack([p, p1row, p2row])[None], (N, 3, V))
    blk_tok = np.broadcast_to(np.array([[[x1], [x2]]], np.int32), (N, 2, 1))
    u_acc = (rng.integers(0, 1 << 24, size=(N, 2, 1)) * 2.0 ** -24).astype(np.float32)
    u_fin = (rng.integers(0, 1 << 24, size=N) * 2.0 ** -24).astype(np.float32)
    r = O.verify_step_accept("sample", "probs_f32", tgt, None, blk_tok, np.ones((N, 2), np.int32), 2, 0,
                             u_acc, u_fin)
    cats = _two_block_categories(p.astype(np.float64), p1row, p2row, x1, x2)
    assert abs(sum(cats.values()) - 1.0) < 1e-6
    keys = list(cats)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys), np.int64)
    for b in range(N):
        n = int(r["n_out"][b])
        key = (int(r["best_blk"][b]), n, int(r["out_tok"][b, 0]), int(r["out_tok"][b, 1]) if n == 2 else -1)
        counts[index[key]] += 1          # a KeyError is an outcome the rules cannot produce
    expected = np.array([cats[k] for k in keys]) * N
    chi2, pval = scipy.stats.chisquare(counts, expected / expected.sum() * N)
    assert pval > 0.01, (chi2, pval)
    # the first emitted token does not follow p: x2 is favoured (p2 (2 - p1 - p2) > p2)
    first = np.bincount(r["out_tok"][:, 0], minlength=V)
    _, pval_p = scipy.stats.chisquare(first, p.astype(np.float64) / p.sum() * N)
    assert pval_p < 1e-6


def test_copy_and_chain_blocks_in_one_step_ties_go_to_the_copy_block():
    """Copy blocks and the chain block verified in one pass (chain block always present):
    the longest run wins and, on a tie, the copy block (the chain block comes last)."""
    V, W, Dmax, K = 8, 2, 3, 3
    NB = W + 1
    eye = np.eye(V, dtype=np.float32)
    tgt = np.tile(eye[1], (1, 1 + NB * Dmax, 1))                    # the target always wants token 1
    drf = np.tile(eye[1], (1, K, 1))
    z = np.zeros((1, NB, Dmax), np.float32)

    def run(copy0, copy1, chain):
        bt = np.array([[copy0, copy1, chain]], np.int32)
        bl = np.array([[3, 3, 3]], np.int32)
        return O.verify_step_accept("greedy", "probs_f32", tgt, drf, bt, bl, W, 2, z, np.zeros(1, np.float32))

    r = run([1, 2, 2], [3, 3, 3], [1, 5, 5])       # copy 0 and chain both accept one token
    assert list(r["acc_len"][0]) == [1, 0, 1] and r["best_blk"][0] == 0
    r = run([1, 2, 2], [3, 3, 3], [1, 1, 1])       # the chain block is longer: it wins
    assert list(r["acc_len"][0]) == [1, 0, 3] and r["best_blk"][0] == 2
    assert r["n_out"][0] == 4 and list(r["out_tok"][0]) == [1, 1, 1, 1]
    r = run([1, 1, 1], [3, 3, 3], [1, 1, 1])       # a full copy block ties the full chain block
    assert r["best_blk"][0] == 0 and list(r["out_tok"][0]) == [1, 1, 1, 1]
