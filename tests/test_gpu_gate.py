"""GPU gate + retrieval against the oracle: bit-exact on every workload shape and
on edge cases (empty, short, periodic and ragged contexts)."""
import numpy as np
import pytest
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import to_device

pytestmark = pytest.mark.gpu


def _run(ctx, ctx_len, h, h_dtype, w, tau, kappa, W, D, K, policy, chain_tok):
    dev = "cuda"
    tc, tl, th, tw = (to_device(np.asarray(a), dev) for a in (ctx, ctx_len, h, w))
    g = S.ssd_gate_match(tc, tl, th, tw, tau, kappa)
    ct = to_device(np.asarray(chain_tok), dev) if policy else None
    r = S.ssd_retrieve(tc, tl, g["gate"], g["last_match_end"], kappa, W, D, K, policy, ct)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in {**g, **r}.items()}


def _run_fused(ctx, ctx_len, h, h_dtype, w, tau, kappa, W, D, K, policy, chain_tok):
    dev = "cuda"
    tc, tl, th, tw = (to_device(np.asarray(a), dev) for a in (ctx, ctx_len, h, w))
    ct = to_device(np.asarray(chain_tok), dev) if policy else None
    r = S.ssd_gate_retrieve(tc, tl, th, tw, tau, kappa, W, D, K, policy, ct)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def _compare(ctx, ctx_len, h, h_dtype, w, tau, kappa, W, D, K, policy, chain_tok):
    got = _run(ctx, ctx_len, h, h_dtype, w, tau, kappa, W, D, K, policy, chain_tok)
    fused = _run_fused(ctx, ctx_len, h, h_dtype, w, tau, kappa, W, D, K, policy, chain_tok)
    for k in got:
        if k == "score":
            np.testing.assert_allclose(fused[k], got[k], atol=1e-6)
        else:
            np.testing.assert_array_equal(fused[k], got[k], err_msg=f"fused {k}")
    score, on, gate, last = O.gate_match(ctx, ctx_len, h, h_dtype, w, tau, kappa)
    bt, bl, nc = O.retrieve(ctx, ctx_len, gate, kappa, W, D, K, policy, chain_tok)
    np.testing.assert_array_equal(got["probe_on"], on.astype(np.int32))
    np.testing.assert_array_equal(got["gate"], gate)
    np.testing.assert_array_equal(got["last_match_end"], last)
    np.testing.assert_allclose(got["score"], score, atol=1e-6)
    np.testing.assert_array_equal(got["blk_len"], bl)
    np.testing.assert_array_equal(got["n_cand"], nc)
    np.testing.assert_array_equal(got["blk_tok"], bt)
    return got


@pytest.mark.parametrize("name", WL.WORKLOAD_ORDER)
@pytest.mark.parametrize("full_width", [True, False])
def test_gate_retrieve_workloads(name, full_width):
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl, 1000 + WL.WORKLOAD_ORDER.index(name), full_width=full_width,
                         with_attention=False, with_logits=False)
    ct = np.random.default_rng(5).integers(0, wl.V, size=(wl.B, wl.K)).astype(np.int32)
    got = _compare(inp["ctx"], inp["ctx_len"], inp["h"], wl.h_dtype, inp["w"], wl.tau, wl.kappa, wl.W, wl.D,
                   wl.K, wl.chain_policy, ct)
    # every sequence whose probe was set high found its planted repeat
    assert np.all(got["gate"][inp["gate_on_target"]] == 1)
    if full_width:
        on = inp["gate_on_target"]
        assert np.all(got["n_cand"][on] == wl.W)


def test_gate_retrieve_edge_cases():
    rng = np.random.default_rng(7)
    lens = [0, 1, 4, 5, 6, 7, 33, 4095, 4096, 4097, 9000, 257]
    B = len(lens)
    stride = max(lens)
    ctx = np.full((B, stride), -1, np.int32)
    for b, n in enumerate(lens):
        kind = b % 3
        if kind == 0:
            row = rng.integers(0, 3, size=n)                 # tiny alphabet: many matches
        elif kind == 1:
            row = np.tile(np.array([9, 8, 7]), n // 3 + 1)[:n]  # periodic
        else:
            row = rng.integers(0, 1 << 20, size=n)           # almost no matches
        ctx[b, :n] = row
    d = 96
    h, w = WL._probe_pair(rng, d, np.linspace(-3, 3, B), "f32")
    for kappa, W, D, K, policy in [(5, 4, 20, 0, 0), (1, 3, 2, 2, 1), (2, 64, 7, 9, 2), (3, 1, 1, 1, 1)]:
        ct = rng.integers(0, 50, size=(B, max(K, 1))).astype(np.int32)[:, :K]
        _compare(ctx, np.array(lens, np.int32), h, "f32", w, 0.4, kappa, W, D, K, policy, ct)
    # tau limits: always on / never on
    for tau in (0.0, 1.0, 0.5):
        _compare(ctx, np.array(lens, np.int32), h, "f32", w, tau, 5, 4, 8, 0, 0, np.zeros((B, 0), np.int32))


def test_gate_threshold_boundary_bit_exact():
    # fixed-point sums exactly at the threshold and one below (the page's "at least tau")
    T = O.probe_threshold_fixed(0.4)
    rows = []
    for target in (T, T - 1, T + 1):
        hi = (target >> 20) << 20
        lo = target - hi
        rows.append([hi * 2.0 ** -32, lo * 2.0 ** -32])
    h = np.array(rows, np.float32)
    w = np.array([1.0, 1.0], np.float32)
    ctx = np.tile(np.array([[1, 2, 1, 2]], np.int32), (3, 1))
    got = _compare(ctx, np.full(3, 4, np.int32), h, "f32", w, 0.4, 1, 2, 2, 0, 0, np.zeros((3, 0), np.int32))
    assert list(got["probe_on"]) == [1, 0, 1]


def test_gate_bf16_random_many_sequences():
    rng = np.random.default_rng(8)
    B, n = 300, 700
    ctx = rng.integers(0, 6, size=(B, n)).astype(np.int32)
    lens = rng.integers(0, n + 1, size=B).astype(np.int32)
    h, w = WL._probe_pair(rng, 4096, rng.normal(size=B) * 0.5, "bf16")
    _compare(ctx, lens, h, "bf16", w, 0.4, 5, 8, 16, 7, 1,
             rng.integers(0, 6, size=(B, 7)).astype(np.int32))
