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
import numpy as np
import pytest

import fullsize_helpers as H
from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300.step import VerifyStep, default_early_rows

pytestmark = pytest.mark.gpu

BIG = ["batched", "llama70b", "qwen8b_mixed", "qwen8b_mixed_act086"]

def test_attention_llama8b_every_token():
    wl, inp = H.inputs("llama8b")
    _, r = H.bench_step(wl, inp)
    bl = r["blk_len"]
    slots = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(int(bl[b, k]))]
    assert len(slots) > 40
    ref = H.oracle_attention(inp, wl, bl, slots)
    assert len(ref) == len(slots)
    assert H.max_err(r["attn"], ref, wl.kv_dtype) <= H.TOL


@pytest.mark.parametrize("name", BIG)
def test_attention_first_row_tile_of_every_sequence(name):
    wl, inp = H.inputs(name)
    _, r = H.bench_step(wl, inp)
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
    ref = H.oracle_attention(inp, wl, bl, slots)
    assert H.max_err(r["attn"], ref, wl.kv_dtype) <= H.TOL


@pytest.mark.parametrize("name", WL.WORKLOAD_ORDER + WL.VARIANT_ORDER)
def test_whole_step_boosted_acceptance(name):
    wl, inp = H.inputs(name)
    pin = H.boosted_probs(wl, {k: v for k, v in inp.items()}, 11 + len(name))
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
