"""Full-size parity through the step's own launch path (the benchmark's configuration:
one stream, the row-pass mode and tile skipping each workload uses).

* Attention of the Llama-3.1-8B-shaped verify: every present token and head against the
  fp64 oracle (max-abs <= 1e-2).
* Attention of the larger shapes: for every sequence, every present token of its first
  128-row tile that holds one (all kv heads) against the oracle.
* Acceptance with long accepted runs: the target rows are boosted (+20 on the verified
  token at a random number of leading positions of every block) and given as fp32
  probabilities, so that copy runs, chain runs, bonus draws and residual draws all occur
  at full size; acceptance, choice and tokens bit-exact against the oracle.
The oracle's attention runs in threads over disjoint slot lists (its numpy work releases
the interpreter lock); each call is the oracle's own function."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300.step import VerifyStep, default_early_rows

pytestmark = pytest.mark.gpu

TOL = 1e-2
BIG = ["batched", "llama70b", "qwen8b_mixed", "qwen8b_mixed_act086"]
_CACHE = {}


def _inputs(name):
    if name not in _CACHE:
        wl = WL.WORKLOADS[name]
        _CACHE[name] = (wl, WL.make_inputs(wl, WL.default_seed(name) + 300, full_width=False))
    return _CACHE[name]


def _oracle_attention(inp, wl, bl, slots, threads=None):
    threads = threads or min(16, os.cpu_count() or 1)
    chunks = [slots[i::threads] for i in range(threads) if slots[i::threads]]
    out = {}
    with cf.ThreadPoolExecutor(len(chunks)) as ex:
        for part in ex.map(lambda ch: O.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"],
                                                         inp["v_cand"], inp["prefix_len"], bl, wl.Dmax, wl.kv_dtype,
                                                         ch), chunks):
            out.update(part)
    return out


def _bench_step(wl, inp, **kw):
    st = VerifyStep(wl, inp, early_rows=default_early_rows(wl), **kw)
    st.run()
    return st, st.results()


def _max_err(got_attn, ref, dtype):
    with np.errstate(invalid="ignore"):
        g = O.to_f64(got_attn, dtype)
    return max(float(np.max(np.abs(g[b, t] - o))) for (b, t), o in ref.items())


def test_attention_llama8b_every_token():
    wl, inp = _inputs("llama8b")
    _, r = _bench_step(wl, inp)
    bl = r["blk_len"]
    slots = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(int(bl[b, k]))]
    assert len(slots) > 40
    ref = _oracle_attention(inp, wl, bl, slots)
    assert len(ref) == len(slots)
    assert _max_err(r["attn"], ref, wl.kv_dtype) <= TOL


@pytest.mark.parametrize("name", BIG)
def test_attention_first_row_tile_of_every_sequence(name):
    wl, inp = _inputs(name)
    _, r = _bench_step(wl, inp)
    bl = r["blk_len"]
    per_tile = 128 // wl.G                   # tokens whose G heads fill one 128-row tile
    slots = []
    for b in range(wl.B):
        present = [k * wl.Dmax + d for k in range(wl.NB) for d in range(int(bl[b, k]))]
        if not present:
            continue
        tile = present[0] // per_tile
        slots += [(b, t) for t in present if t // per_tile == tile]
    assert {b for b, _ in slots} == {b for b in range(wl.B) if bl[b].sum() > 0}
    ref = _oracle_attention(inp, wl, bl, slots)
    assert _max_err(r["attn"], ref, wl.kv_dtype) <= TOL


def _boosted_probs(wl, inp, seed):
    """Target and draft rows as fp32 probabilities (the oracle's softmax), the target rows
    boosted so that each block accepts a random number of leading tokens."""
    kind = "logits_bf16" if wl.logit_dtype == "bf16" else "logits_f32"
    _, _, gate, _ = O.gate_match(inp["ctx"], inp["ctx_len"], inp["h"], wl.h_dtype, inp["w"], wl.tau, wl.kappa)
    bt, bl, _ = O.retrieve(inp["ctx"], inp["ctx_len"], gate, wl.kappa, wl.W, wl.D, wl.K, wl.chain_policy,
                           inp["chain_tok"])
    rng = np.random.default_rng(seed)
    rows = {}
    for b in range(wl.B):
        for k in range(wl.NB):
            # every third block accepts all of its tokens (bonus draws), the others a random run
            a = int(bl[b, k]) if (b + k) % 3 == 0 else int(rng.integers(0, int(bl[b, k]) + 1))
            for d in range(a):
                rows[(b, 0 if d == 0 else 1 + k * wl.Dmax + d - 1)] = int(bt[b, k, d])
    tgt = WL.boost_accepts(inp["tgt"], wl.logit_dtype, rows)
    out = dict(inp)
    out["tgt"] = np.stack([O.row_probs(tgt[b], kind) for b in range(wl.B)])
    if inp.get("drf") is not None:
        out["drf"] = np.stack([O.row_probs(inp["drf"][b], kind) for b in range(wl.B)])
    return out


@pytest.mark.parametrize("name", WL.WORKLOAD_ORDER + WL.VARIANT_ORDER)
def test_whole_step_boosted_acceptance(name):
    wl, inp = _inputs(name)
    pin = _boosted_probs(wl, {k: v for k, v in inp.items()}, 11 + len(name))
    st = VerifyStep(wl, pin, kind=S.SSD_PROBS_F32, with_attention=False, early_rows=default_early_rows(wl))
    for _ in range(2):                       # the second run's results are checked
        st.run()
    got = st.results()
    ref = O.verify_step(pin, wl, attention_slots=None, kind="probs_f32")
    for k in ("gate", "blk_tok", "blk_len", "n_cand", "acc_len", "best_blk", "n_out", "out_tok"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    # the boost produced long runs and both kinds of final draw
    a = ref["n_out"] - 1
    L = np.array([ref["blk_len"][b, k] if k >= 0 else 0 for b, k in enumerate(ref["best_blk"])])
    assert a.max() >= 5
    if wl.B > 1:
        assert np.any((a == L) & (L > 0)) and np.any(a < L)
