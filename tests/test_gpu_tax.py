"""Copy attempts and the speculation tax on the GPU against the oracle counts, on a
batch where every sequence ends in a repeated 5-gram: half copy-intended (probe high,
the target follows the copy), half accidental (probe low, unrelated target). The
surface gate (tau = 0) opens every copy and pays the tax on the accidental half; the
probe gate opens only the intended ones."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import VerifyStep

pytestmark = pytest.mark.gpu


def tax_inputs(seed=5):
    wl = WL.TAX_WORKLOAD
    B = wl.B
    intended = np.zeros(B, bool)
    intended[::2] = True
    inp = WL.make_inputs(wl, seed, with_attention=False, gate_on=np.ones(B, bool), probe_on=intended)
    # the target follows the copy of the intended sequences: boost each candidate token of
    # every block on the row that verifies it
    ref = O.verify_step(dict(inp), dataclasses.replace(wl, tau=0.0), attention_slots=None)
    rows = {}
    for b in np.flatnonzero(intended):
        for k in range(wl.NB):
            for d in range(int(ref["blk_len"][b, k])):
                r = 0 if d == 0 else 1 + k * wl.Dmax + d - 1
                rows[(int(b), r)] = int(ref["blk_tok"][b, k, d])
    inp["tgt"] = WL.boost_accepts(inp["tgt"], wl.logit_dtype, rows)
    return wl, inp, intended


@pytest.mark.parametrize("tau", [0.0, 0.4])
def test_copy_stats_surface_vs_probe(tau):
    wl0, inp, intended = tax_inputs()
    wl = dataclasses.replace(wl0, tau=tau)
    st = VerifyStep(wl, inp, with_attention=False)
    counts = torch.zeros(4, dtype=torch.int64, device="cuda")
    st.run()
    S.ssd_copy_stats(st.gate_out["gate"], st.ret_out["n_cand"], st.acc_out["acc_len"], wl.W, counts)
    got = counts.cpu().numpy()
    r = st.results()
    ref = O.copy_stats(r["gate"], r["n_cand"], r["acc_len"], wl.W)
    np.testing.assert_array_equal(got, ref)
    oref = O.verify_step(inp, wl, attention_slots=None)
    np.testing.assert_array_equal(r["gate"], oref["gate"])
    B = wl.B
    if tau == 0.0:
        assert got[0] == B                      # every repeat opens a copy
        assert got[1] >= B // 2 - 2             # the accidental half pays the tax
    else:
        assert got[0] == intended.sum()         # only the intended copies open
        assert got[1] <= 2                      # and they are accepted
    assert got[3] == B
