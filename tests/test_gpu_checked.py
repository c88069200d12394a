"""The checked build (libssd_checked.so, -DSSD_CHECKS=1): every guarded device index is
tested before the access. The step of each of the five workloads runs through it with
canary regions around every output and workspace buffer; results match the oracle, no
device error or check failure is recorded and every canary is intact. Out-of-range
lengths (a context length past its row, a prefix length past the cache) are reported
by the checked build instead of being read."""
import numpy as np
import pytest
import torch

import fullsize_helpers as H
from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import VerifyStep, default_early_rows, to_device

pytestmark = pytest.mark.gpu

GUARD = 4096                    # bytes of canary before and after every buffer
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    with S.use_library(S.CHECKED_LIB_PATH) as L:
        assert L.ssd_checked_build() == 1
        S.ssd_read_check_error()                 # start from clear check words
        yield


class Guarded:
    """Buffers with canary regions on both sides; views of them stand in for outputs."""

    def __init__(self):
        self.bufs = []

    def like(self, t):
        n = t.numel() * t.element_size()
        raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=t.device)
        view = raw[GUARD:GUARD + n].view(t.dtype).view(t.shape)
        view.copy_(t)
        self.bufs.append(raw)
        return view

    def intact(self):
        torch.cuda.synchronize()
        for raw in self.bufs:
            g = torch.cat([raw[:GUARD], raw[-GUARD:]])
            if not bool((g == PATTERN).all()):
                return False
        return True


def _guard_step(st, G):
    for d in (st.gate_out, st.ret_out, st.acc_out):
        for k in d:
            d[k] = G.like(d[k])
    st.acc_ws = G.like(st.acc_ws)
    if st.with_attention:
        st.attn_out = G.like(st.attn_out)
        st.attn_ws = G.like(st.attn_ws)


@pytest.mark.parametrize("name", WL.WORKLOAD_ORDER)
def test_checked_step_with_canaries(name):
    wl, inp = H.inputs(name)
    pin = H.boosted_probs(wl, dict(inp), 21 + len(name))
    pin = {**inp, "tgt": pin["tgt"], "drf": pin["drf"]}
    st = VerifyStep(wl, pin, kind=S.SSD_PROBS_F32, early_rows=default_early_rows(wl))
    G = Guarded()
    _guard_step(st, G)
    st.run()
    got = st.results()
    assert G.intact(), "a canary region was written"
    assert S.ssd_read_device_error(st.acc_ws) == S.SSD_OK
    if st.with_attention:
        assert S.ssd_read_device_error(st.attn_ws) == S.SSD_OK
    assert S.ssd_read_check_error() == S.SSD_OK
    ref = O.verify_step(pin, wl, attention_slots=None, kind="probs_f32")
    for k in ("gate", "blk_tok", "blk_len", "n_cand", "acc_len", "best_blk", "n_out", "out_tok"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    bl = ref["blk_len"]
    slots = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(int(bl[b, k]))][:48]
    ra = H.oracle_attention(inp, wl, bl, slots)
    assert H.max_err(got["attn"], ra, wl.kv_dtype) <= H.TOL


def test_checked_build_reports_a_context_length_past_its_row():
    wl = WL.WORKLOADS["tiny"]
    inp = WL.make_inputs(wl, 3, with_attention=False, with_logits=False)
    dev = "cuda"
    ctx, ctx_len = to_device(inp["ctx"], dev), to_device(inp["ctx_len"], dev)
    ctx_len[0] = ctx.shape[1] + 7                  # past the row: the checked build reads nothing
    out = S.ssd_gate_match(ctx, ctx_len, to_device(inp["h"], dev), to_device(inp["w"], dev), wl.tau, wl.kappa)
    torch.cuda.synchronize()
    assert S.ssd_read_check_error() == S.SSD_ERR_DEVICE
    assert int(out["last_match_end"][0]) == -1 and int(out["gate"][0]) == 0
    assert S.ssd_read_check_error() == S.SSD_OK


def test_checked_build_reports_a_prefix_past_the_cache():
    rng = np.random.default_rng(4)
    B, NB, Dmax, Hkv, G, dh, P = 1, 2, 4, 2, 4, 128, 256
    f = lambda *s: WL.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    dev = "cuda"
    T = lambda a: to_device(a, dev)
    q, kc, vc = T(f(B, NB * Dmax, Hkv * G, dh)), T(f(B, Hkv, P, dh)), T(f(B, Hkv, P, dh))
    kd, vd = T(f(B, NB * Dmax, Hkv, dh)), T(f(B, NB * Dmax, Hkv, dh))
    pl, bl = T(np.array([P + 100], np.int32)), T(np.full((B, NB), Dmax, np.int32))
    out = torch.empty_like(q)
    ws = torch.zeros(S.ssd_verify_attn_workspace_size(S.attn_args(q, kc, vc, kd, vd, pl, bl, Dmax, out)),
                     dtype=torch.uint8, device=dev)
    S.ssd_verify_attn(q, kc, vc, kd, vd, pl, bl, Dmax, out=out, ws=ws)
    assert S.ssd_read_device_error(ws) == S.SSD_ERR_DEVICE
    assert S.ssd_read_check_error() == S.SSD_ERR_DEVICE
