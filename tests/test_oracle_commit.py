"""Pins of the oracle's commit of accepted keys/values (anatomy page §6, KV cache
rollback): what the commit leaves in the cache must reproduce the verification
attention of the accepted tokens, nothing else may change, and the prefix grows
by exactly the accepted count of a real acceptance step."""
import numpy as np
import torch

from oracle import ssd_oracle as O


def _case(rng, B, NB, Dmax, Hq, Hkv, dh, P_max, prefix):
    NT = NB * Dmax
    f = lambda *s: rng.standard_normal(s)
    return dict(q=f(B, NT, Hq, dh), k_cache=f(B, Hkv, P_max, dh), v_cache=f(B, Hkv, P_max, dh),
                k_cand=f(B, NT, Hkv, dh), v_cand=f(B, NT, Hkv, dh), prefix_len=np.asarray(prefix, np.int32))


def _plain_attention(q, keys, vals):
    """softmax(q k^T / sqrt(dh)) v for one kv head's q rows, fp64, by torch's SDPA."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(keys), t(vals))
    return o[0, 0].numpy()


def test_committed_cache_reproduces_verification():
    """Token d of the chosen block attended, when verified, to the prefix and its own
    block's tokens 1..d; after the commit the same query over cache rows [0, P+d)
    must give the same output: right slots, right order, every kv head."""
    rng = np.random.default_rng(11)
    B, NB, Dmax, Hq, Hkv, dh, P_max = 3, 3, 6, 4, 2, 16, 40
    c = _case(rng, B, NB, Dmax, Hq, Hkv, dh, P_max, [0, 13, 20])
    blk_len = np.array([[6, 2, 0], [3, 6, 5], [1, 1, 6]], np.int32)
    best = np.array([0, 1, 2], np.int32)
    n_out = np.array([7, 5, 3], np.int32)                 # a = 6, 4, 2 accepted
    ref = O.verify_attention(c["q"], c["k_cache"], c["v_cache"], c["k_cand"], c["v_cand"], c["prefix_len"],
                             blk_len, Dmax, "f32")
    kc, vc, pl, ok = O.commit_kv(c["k_cache"], c["v_cache"], c["k_cand"], c["v_cand"], c["prefix_len"], best,
                                 n_out, Dmax)
    assert ok.all()
    np.testing.assert_array_equal(pl, c["prefix_len"] + n_out - 1)
    G = Hq // Hkv
    for b in range(B):
        k, a, P = int(best[b]), int(n_out[b]) - 1, int(c["prefix_len"][b])
        for d in range(1, a + 1):
            t = k * Dmax + d - 1
            for kvh in range(Hkv):
                q = c["q"][b, t, kvh * G:(kvh + 1) * G].astype(np.float32).astype(np.float64)
                o = _plain_attention(q, kc[b, kvh, :P + d].astype(np.float32).astype(np.float64),
                                     vc[b, kvh, :P + d].astype(np.float32).astype(np.float64))
                np.testing.assert_allclose(o, ref[(b, t)][kvh * G:(kvh + 1) * G], rtol=1e-10, atol=1e-12)
        # nothing outside the new rows changed
        np.testing.assert_array_equal(kc[b, :, :P], c["k_cache"][b, :, :P])
        np.testing.assert_array_equal(kc[b, :, P + a:], c["k_cache"][b, :, P + a:])
        np.testing.assert_array_equal(vc[b, :, P + a:], c["v_cache"][b, :, P + a:])


def test_nothing_committed_cases():
    rng = np.random.default_rng(12)
    c = _case(rng, 3, 2, 4, 2, 1, 8, 10, [3, 9, 5])
    best = np.array([-1, 0, 1], np.int32)
    n_out = np.array([1, 3, 1], np.int32)                 # no block; no room (9 + 2 > 10); a = 0
    kc, vc, pl, ok = O.commit_kv(c["k_cache"], c["v_cache"], c["k_cand"], c["v_cand"], c["prefix_len"], best,
                                 n_out, 4)
    np.testing.assert_array_equal(kc, c["k_cache"])
    np.testing.assert_array_equal(vc, c["v_cache"])
    np.testing.assert_array_equal(pl, c["prefix_len"])
    assert list(ok) == [True, False, True]


def test_prefix_grows_by_the_greedy_common_prefix():
    """Greedy verification accepts a block's tokens while each equals the target's own
    choice at that position (the greedy page, "2단계 · 일괄 검증"): the longest such run
    over the blocks, found here by a plain scan, is what the commit appends."""
    rng = np.random.default_rng(13)
    B, W, Dmax, V = 4, 3, 5, 7
    for rep in range(20):
        blk_tok = rng.integers(0, V, size=(B, W, Dmax)).astype(np.int32)
        blk_len = rng.integers(1, Dmax + 1, size=(B, W)).astype(np.int32)
        tgt = rng.random((B, 1 + W * Dmax, V)).astype(np.float32)
        # often make the target agree with the candidate, so that runs are long
        for b in range(B):
            for k in range(W):
                for d in range(Dmax):
                    r = 0 if d == 0 else 1 + k * Dmax + d - 1
                    if rng.random() < 0.7:
                        tgt[b, r, blk_tok[b, k, d]] = 2.0
        res = O.verify_step_accept("greedy", "logits_f32", tgt, None, blk_tok, blk_len, W, 0,
                                   np.zeros((B, W, Dmax), np.float32), np.zeros(B, np.float32))
        run = np.zeros((B, W), np.int64)
        for b in range(B):
            for k in range(W):
                for d in range(int(blk_len[b, k])):
                    r = 0 if d == 0 else 1 + k * Dmax + d - 1
                    if int(np.argmax(tgt[b, r])) != int(blk_tok[b, k, d]):
                        break
                    run[b, k] += 1
        longest = run.max(axis=1)
        c = _case(rng, B, W, Dmax, 2, 1, 4, 64, [7, 30, 0, 50])
        kc, vc, pl, ok = O.commit_kv(c["k_cache"], c["v_cache"], c["k_cand"], c["v_cand"], c["prefix_len"],
                                     res["best_blk"], res["n_out"], Dmax)
        assert ok.all()
        np.testing.assert_array_equal(pl, c["prefix_len"] + longest)
