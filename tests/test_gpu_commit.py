"""GPU commit of accepted keys/values against the oracle: bit-exact caches and
prefix lengths (bf16 and fp32, aligned and unaligned rows), sequences without a
block, without room, or with nothing accepted; and after a whole GPU step."""
import numpy as np
import pytest
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import VerifyStep, to_device

pytestmark = pytest.mark.gpu


def _arrays(rng, B, NB, Dmax, Hkv, dh, P_max, dtype):
    NT = NB * Dmax
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    cast = (lambda x: x) if dtype == "f32" else WL.f32_to_bf16_bits
    return dict(k_cache=cast(f(B, Hkv, P_max, dh)), v_cache=cast(f(B, Hkv, P_max, dh)),
                k_cand=cast(f(B, NT, Hkv, dh)), v_cand=cast(f(B, NT, Hkv, dh)))


@pytest.mark.parametrize("dtype,dh", [("bf16", 128), ("f32", 64), ("bf16", 5), ("f32", 3)])
def test_commit_matches_oracle(dtype, dh):
    rng = np.random.default_rng(dh + len(dtype))
    B, NB, Dmax, Hkv, P_max = 6, 3, 7, 2, 40
    c = _arrays(rng, B, NB, Dmax, Hkv, dh, P_max, dtype)
    prefix = np.array([0, 10, 39, 20, 34, 5], np.int32)
    best = np.array([0, 2, 1, -1, 1, 2], np.int32)
    n_out = np.array([8, 4, 2, 1, 8, 1], np.int32)      # a = 7, 3, 1 (exactly fills), 0, 7 (no room), 0
    kc, vc, pl, ok = O.commit_kv(c["k_cache"], c["v_cache"], c["k_cand"], c["v_cand"], prefix, best, n_out, Dmax)
    t = {k: to_device(v, "cuda") for k, v in c.items()}
    pl_d = to_device(prefix, "cuda")
    ws = S.ssd_commit_kv(t["k_cache"], t["v_cache"], t["k_cand"], t["v_cand"], pl_d, to_device(best, "cuda"),
                         to_device(n_out, "cuda"), Dmax)
    torch.cuda.synchronize()
    as_np = lambda x: x.cpu().numpy().view(np.uint16) if dtype == "bf16" else x.cpu().numpy()
    np.testing.assert_array_equal(as_np(t["k_cache"]), kc)
    np.testing.assert_array_equal(as_np(t["v_cache"]), vc)
    np.testing.assert_array_equal(pl_d.cpu().numpy(), pl)
    assert S.ssd_read_device_error(ws) == (S.SSD_OK if ok.all() else S.SSD_ERR_DEVICE)
    assert not ok[4]


def test_commit_after_a_gpu_step():
    """The step's own outputs drive the commit: a cache with room past the prefix grows by
    the accepted run of the chosen block and holds exactly those candidate rows."""
    wl = WL.WORKLOADS["llama8b"]
    inp = WL.make_inputs(wl, 99, full_width=False)
    # accepted runs: the target logit of a leading candidate token raised by 20
    ref = O.verify_step(inp, wl, attention_slots=None)
    rng = np.random.default_rng(7)
    tgt = np.array(inp["tgt"], copy=True)
    for b in range(wl.B):
        for k in range(wl.NB):
            for d in range(int(rng.integers(0, ref["blk_len"][b, k] + 1))):
                r = 0 if d == 0 else 1 + k * wl.Dmax + d - 1
                tgt[b, r, ref["blk_tok"][b, k, d]] += 20.0
    inp = dict(inp, tgt=tgt)
    st = VerifyStep(wl, inp)
    st.run()
    got = st.results()
    B, Hkv, P_max, dh = st.x["k_cache"].shape
    room = wl.NB * wl.Dmax
    kb = torch.zeros((B, Hkv, P_max + room, dh), dtype=st.x["k_cache"].dtype, device="cuda")
    vb = torch.zeros_like(kb)
    kb[:, :, :P_max] = st.x["k_cache"]
    vb[:, :, :P_max] = st.x["v_cache"]
    k0, v0 = kb.cpu().numpy().view(np.uint16), vb.cpu().numpy().view(np.uint16)
    pre = st.x["prefix_len"].clone()
    ws = S.ssd_commit_kv(kb, vb, st.x["k_cand"], st.x["v_cand"], st.x["prefix_len"], st.acc_out["best_blk"],
                         st.acc_out["n_out"], wl.Dmax)
    torch.cuda.synchronize()
    assert S.ssd_read_device_error(ws) == S.SSD_OK
    kc, vc, pl, ok = O.commit_kv(k0, v0, inp["k_cand"], inp["v_cand"], pre.cpu().numpy(), got["best_blk"],
                                 got["n_out"], wl.Dmax)
    assert ok.all() and (pl > pre.cpu().numpy()).any()
    np.testing.assert_array_equal(st.x["prefix_len"].cpu().numpy(), pl)
    np.testing.assert_array_equal(kb.cpu().numpy().view(np.uint16), kc)
    np.testing.assert_array_equal(vb.cpu().numpy().view(np.uint16), vc)
