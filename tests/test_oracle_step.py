"""The oracle's whole step on the small workload: structural invariants that
any correct step satisfies (no GPU)."""
import numpy as np

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL


def test_tiny_step_invariants():
    wl = WL.WORKLOADS["tiny"]
    for seed, full in [(None, True), (11, False), (12, False)]:
        inp = WL.make_inputs(wl, seed, full_width=full)
        r = O.verify_step(inp, wl)
        assert r["gate"][0] == 1                       # probe score 0.9 and a planted repeat
        assert 1 <= r["n_cand"][0] <= wl.W
        if full:
            assert r["n_cand"][0] == wl.W and all(r["blk_len"][0, :wl.W] == wl.D)
        k = r["best_blk"][0]
        a = r["acc_len"][0, k]
        assert r["n_out"][0] == a + 1
        assert list(r["out_tok"][0, :a]) == list(r["blk_tok"][0, k, :a])
        assert 0 <= r["out_tok"][0, a] < wl.V
        for o in r["attn"].values():
            assert np.all(np.isfinite(o))
        # each copy candidate is the continuation of an earlier occurrence
        n = int(inp["ctx_len"][0])
        ctx = inp["ctx"][0]
        for kk in range(r["n_cand"][0]):
            L = r["blk_len"][0, kk]
            toks = r["blk_tok"][0, kk, :L]
            starts = [j for j in range(n - L) if list(ctx[j:j + L]) == list(toks)]
            assert starts


def test_gate_off_takes_chain_block():
    wl = WL.WORKLOADS["tiny"]
    inp = WL.make_inputs(wl, 21, gate_on=[False])
    r = O.verify_step(inp, wl)
    assert r["gate"][0] == 0 and r["n_cand"][0] == 0
    assert list(r["blk_len"][0]) == [0, 0, wl.K]
    assert r["best_blk"][0] == wl.W
