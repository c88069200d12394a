"""Pins of the oracle's verification attention against a library routine
(torch scaled_dot_product_attention with an explicitly built mask), the
block-isolation invariant and textbook special cases (no GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL


def _rand_case(seed, B=2, NB=3, Dmax=4, Hq=4, Hkv=2, dh=16, P=(7, 0), dtype="f32"):
    rng = np.random.default_rng(seed)
    P_max = max(max(P), 1)
    NT = NB * Dmax
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    cast = (lambda x: x) if dtype == "f32" else WL.f32_to_bf16_bits
    case = dict(q=cast(f(B, NT, Hq, dh) * 2), k_cache=cast(f(B, Hkv, P_max, dh)),
                v_cache=cast(f(B, Hkv, P_max, dh)), k_cand=cast(f(B, NT, Hkv, dh)),
                v_cand=cast(f(B, NT, Hkv, dh)), prefix_len=np.array(P[:B], dtype=np.int32))
    blk_len = rng.integers(0, Dmax + 1, size=(B, NB)).astype(np.int32)
    blk_len[:, 0] = Dmax
    return case, blk_len


def _sdpa_reference(case, blk_len, Dmax, dtype):
    """Materialise the key sequence [prefix ; every candidate slot] and the
    block-triangular mask from its definition, then call the library routine."""
    q, kc, vc, kd, vd = (O.to_f64(case[n], dtype) for n in ("q", "k_cache", "v_cache", "k_cand", "v_cand"))
    B, NT, Hq, dh = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = {}
    for b in range(B):
        P = int(case["prefix_len"][b])
        keys = np.concatenate([kc[b, :, :P], kd[b].transpose(1, 0, 2)], axis=1)   # [Hkv][P+NT][dh]
        vals = np.concatenate([vc[b, :, :P], vd[b].transpose(1, 0, 2)], axis=1)
        mask = np.zeros((NT, P + NT), dtype=bool)
        for t in range(NT):
            mask[t, :P] = True                           # the whole prefix
            k, pos = divmod(t, Dmax)
            for s in range(NT):
                ks, ps = divmod(s, Dmax)
                mask[t, P + s] = (ks == k) and (ps <= pos)   # own block, earlier or self
        qt = torch.from_numpy(q[b].transpose(1, 0, 2).copy())              # [Hq][NT][dh]
        kt = torch.from_numpy(np.repeat(keys, G, axis=0))                  # [Hq][P+NT][dh]
        vt = torch.from_numpy(np.repeat(vals, G, axis=0))
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))
        o = o.numpy().transpose(1, 0, 2)                                   # [NT][Hq][dh]
        for k in range(blk_len.shape[1]):
            for d in range(1, int(blk_len[b, k]) + 1):
                out[(b, k * Dmax + d - 1)] = o[k * Dmax + d - 1]
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attention_matches_library_with_explicit_mask(seed, dtype):
    case, blk_len = _rand_case(seed, dtype=dtype)
    Dmax = 4
    got = O.verify_attention(case["q"], case["k_cache"], case["v_cache"], case["k_cand"], case["v_cand"],
                             case["prefix_len"], blk_len, Dmax, dtype)
    ref = _sdpa_reference(case, blk_len, Dmax, dtype)
    assert set(got) == set(ref)
    for key in ref:
        np.testing.assert_allclose(got[key], ref[key], rtol=0, atol=1e-12)


def test_block_isolation_invariant():
    # the output of block k equals plain causal attention over prefix || block k alone
    case, blk_len = _rand_case(5, B=1, NB=3, Dmax=5, P=(9,))
    Dmax = 5
    full = O.verify_attention(case["q"], case["k_cache"], case["v_cache"], case["k_cand"], case["v_cand"],
                              case["prefix_len"], blk_len, Dmax, "f32")
    for k in range(3):
        sl = slice(k * Dmax, (k + 1) * Dmax)
        one = O.verify_attention(case["q"][:, sl], case["k_cache"], case["v_cache"], case["k_cand"][:, sl],
                                 case["v_cand"][:, sl], case["prefix_len"], blk_len[:, k:k + 1], Dmax, "f32")
        for (b, t), o in one.items():
            np.testing.assert_allclose(full[(b, k * Dmax + t)], o, rtol=0, atol=1e-13)


def test_no_prefix_is_causal_self_attention():
    case, blk_len = _rand_case(9, B=1, NB=1, Dmax=6, P=(0,))
    blk_len[:] = 6
    got = O.verify_attention(case["q"], case["k_cache"], case["v_cache"], case["k_cand"], case["v_cand"],
                             case["prefix_len"], blk_len, 6, "f32")
    q = torch.from_numpy(case["q"][0].astype(np.float64).transpose(1, 0, 2).copy())
    k = torch.from_numpy(np.repeat(case["k_cand"][0].astype(np.float64).transpose(1, 0, 2), 2, axis=0).copy())
    v = torch.from_numpy(np.repeat(case["v_cand"][0].astype(np.float64).transpose(1, 0, 2), 2, axis=0).copy())
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True).numpy().transpose(1, 0, 2)
    for t in range(6):
        np.testing.assert_allclose(got[(0, t)], ref[t], atol=1e-12)


def test_special_cases():
    rng = np.random.default_rng(11)
    B, NB, Dmax, Hq, Hkv, dh, P = 1, 2, 3, 2, 1, 8, 5
    NT = NB * Dmax
    q = rng.standard_normal((B, NT, Hq, dh)).astype(np.float32)
    kc = np.tile(rng.standard_normal((1, 1, 1, dh)).astype(np.float32), (B, Hkv, P, 1))
    kd = np.tile(kc[:, :1, :1], (1, NT, 1, 1)).reshape(B, NT, Hkv, dh)
    vc = rng.standard_normal((B, Hkv, P, dh)).astype(np.float32)
    vd = rng.standard_normal((B, NT, Hkv, dh)).astype(np.float32)
    bl = np.array([[3, 2]], dtype=np.int32)
    # all keys equal -> uniform weights -> mean of the allowed values
    got = O.verify_attention(q, kc, vc, kd, vd, np.array([P]), bl, Dmax, "f32")
    for (b, t), o in got.items():
        k, pos = divmod(t, Dmax)
        allowed = np.concatenate([vc[0, 0], vd[0, k * Dmax:k * Dmax + pos + 1, 0]]).astype(np.float64)
        np.testing.assert_allclose(o, np.tile(allowed.mean(axis=0), (Hq, 1)), atol=1e-12)
    # one key with an overwhelming score returns its value row
    kc2 = np.zeros((B, Hkv, P, dh), np.float32)
    kd2 = np.zeros((B, NT, Hkv, dh), np.float32)
    q2 = np.zeros((B, NT, Hq, dh), np.float32)
    q2[..., 0] = 1.0
    kc2[0, 0, 3, 0] = 1e4
    got = O.verify_attention(q2, kc2, vc, kd2, vd, np.array([P]), bl, Dmax, "f32")
    for o in got.values():
        np.testing.assert_allclose(o, np.tile(vc[0, 0, 3].astype(np.float64), (Hq, 1)), atol=1e-12)
    # single token, no prefix: its own value
    got = O.verify_attention(q[:, :1], kc[:, :, :0], vc[:, :, :0], kd[:, :1], vd[:, :1],
                             np.array([0]), np.array([[1]], np.int32), 1, "f32")
    np.testing.assert_allclose(got[(0, 0)], np.tile(vd[0, 0, 0].astype(np.float64), (Hq, 1)), atol=1e-12)
