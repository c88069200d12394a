"""The seeded input generator against the recipe it states: determinism, the probe
scores, the Zipf head, planted repeats, the gated-off share, the logit variance and the
uniforms (no GPU). The generator holds none of the step's arithmetic; these tests check
that the inputs have the structure the workloads are described with."""
import math

import numpy as np
import pytest

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL


def test_inputs_are_seeded_and_reproducible():
    wl = WL.WORKLOADS["tiny"]
    a, b = WL.make_inputs(wl, 5), WL.make_inputs(wl, 5)
    c = WL.make_inputs(wl, 6)
    for k in ("ctx", "h", "w", "q", "k_cache", "tgt", "drf", "u_acc", "u_fin"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    assert not np.array_equal(a["ctx"], c["ctx"]) and not np.array_equal(a["tgt"], c["tgt"])


@pytest.mark.parametrize("name", ["tiny", "llama8b", "batched", "llama70b", "qwen8b_mixed"])
def test_probe_scores_are_the_targets(name):
    """h = alpha w/|w|^2 + noise orthogonal to w gives sigma(w.h) = 0.9 (on) or 0.1 (off),
    up to the rounding of h to its storage type."""
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl, 3, with_attention=False, with_logits=False)
    h = O.to_f64(inp["h"], wl.h_dtype)
    s = 1.0 / (1.0 + np.exp(-(h @ inp["w"].astype(np.float64))))
    want = np.where(inp["gate_on_target"], 0.9, 0.1)
    np.testing.assert_allclose(s, want, atol=0.01)
    assert inp["gate_on_target"].sum() == round(wl.gate_on_frac * wl.B)


def test_zipf_sampler_head_follows_the_power_law():
    rng = np.random.default_rng(1)
    V, s, n = 128256, 1.1, 1_000_000
    perm = np.arange(V, dtype=np.int32)                  # identity: ids are ranks - 1
    ids = WL._zipf_ids(rng, n, V, s, perm)
    H = float(np.sum(np.arange(1, V + 1, dtype=np.float64) ** -s))
    counts = np.bincount(ids, minlength=V)
    for k in (1, 2, 3, 10):
        p = k ** -s / H
        assert abs(counts[k - 1] / n - p) < 4 * math.sqrt(p * (1 - p) / n), k


def test_planted_repeats_cover_about_the_stated_density():
    """Llama-3.1-8B shape: about 30% of the context lies in verbatim copies of spans of
    20-200 tokens. Positions whose 12-gram occurred earlier measure it (accidental 12-gram
    repeats of Zipf text over 128k ids do not occur at this length)."""
    wl = WL.WORKLOADS["llama8b"]
    inp = WL.make_inputs(wl, 7, with_attention=False, with_logits=False)
    row = inp["ctx"][0, :int(inp["ctx_len"][0])]
    seen, hit = set(), 0
    for j in range(11, len(row)):
        g = tuple(row[j - 11:j + 1])
        hit += g in seen
        seen.add(g)
    frac = hit / len(row)
    assert 0.18 <= frac <= 0.40, frac
    # the uniform-text workload plants exactly its four spans and nothing repeats by chance
    t = WL.WORKLOADS["tiny"]
    tin = WL.make_inputs(t, 7, with_attention=False, with_logits=False, gate_on=[False])
    r = tin["ctx"][0]
    seen, hit = set(), 0
    for j in range(7, len(r)):
        g = tuple(r[j - 7:j + 1])
        hit += g in seen
        seen.add(g)
    assert 0 < hit <= 4 * (40 - 7)


def test_full_width_gate_on_sequences_give_w_full_candidates():
    wl = WL.WORKLOADS["llama8b"]
    inp = WL.make_inputs(wl, with_attention=False, with_logits=False)
    _, _, gate, _ = O.gate_match(inp["ctx"], inp["ctx_len"], inp["h"], wl.h_dtype, inp["w"], wl.tau, wl.kappa)
    _, blk_len, n_cand = O.retrieve(inp["ctx"], inp["ctx_len"], gate, wl.kappa, wl.W, wl.D, wl.K,
                                    wl.chain_policy, inp["chain_tok"])
    assert gate[0] == 1 and n_cand[0] == wl.W
    assert list(blk_len[0, :wl.W]) == [wl.D] * wl.W


def test_logits_have_the_stated_variance_and_uniforms_are_exact():
    wl = WL.WORKLOADS["llama8b"]
    inp = WL.make_inputs(wl, 9, with_attention=False)
    x = inp["tgt"].astype(np.float64).ravel()
    assert abs(x.mean()) < 0.01 and abs(x.var() - 3.0) < 0.03            # N(0, 3): 3 is the variance
    t = WL.make_inputs(WL.WORKLOADS["tiny"], 9, with_attention=False)
    assert abs(t["tgt"].astype(np.float64).var() - 2.0) < 0.05
    for u in (inp["u_acc"], inp["u_fin"], t["u_acc"]):
        k = u.astype(np.float64) * 2.0 ** 24
        assert np.all(k == np.floor(k)) and u.min() >= 0.0 and u.max() < 1.0
