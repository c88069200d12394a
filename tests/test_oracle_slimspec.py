"""Pins of the SlimSpec head oracle (SlimSpec page, "방법론: SlimSpec" / "아키텍처":
z = W_up W_down h; the draft distribution q = softmax(z)) against a hand-worked
case, special cases that reduce to plain selections, brute force on tiny
integer inputs, closed forms of the log-sum-exp and a library routine."""
import json
import math
import os

import numpy as np
import pytest

from oracle import slimspec_oracle as S
from speculative_decoding_copy_gb300.workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "slimspec_tiny.json")


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def test_hand_worked_case():
    g = json.load(open(GOLDEN))
    out = S.slimspec_head(_bits(g["h"]), _bits(g["w_down"]), _bits(g["w_up"]))
    np.testing.assert_array_equal(out["u"], g["u"])
    np.testing.assert_array_equal(out["z"], g["z"])
    np.testing.assert_array_equal(out["row_max"], g["row_max"])
    np.testing.assert_array_equal(out["argmax"], g["argmax"])
    lse = [eval(e, {"log": math.log, "exp": math.exp}) for e in g["lse_closed_form"]]
    np.testing.assert_allclose(out["lse"], lse, rtol=0, atol=1e-14)
    # the factored head gives the full-rank head's logits for W_full = W_up W_down
    full = S.fullrank_head(_bits(g["h"]), _bits(g["w_full"]))
    np.testing.assert_array_equal(full["z"], g["z"])
    np.testing.assert_array_equal(full["argmax"], g["argmax"])


def test_brute_force_tiny_integers():
    rng = np.random.default_rng(5)
    M, d, r, V = 3, 7, 3, 11
    h = rng.integers(-4, 5, (M, d)).astype(np.float64)
    wd = rng.integers(-3, 4, (r, d)).astype(np.float64)
    wu = rng.integers(-3, 4, (V, r)).astype(np.float64)
    u, z = S.lowrank_project(h, wd, wu)
    for m in range(M):
        for v in range(V):
            acc = 0
            for j in range(r):
                inner = 0
                for k in range(d):
                    inner += int(wd[j, k]) * int(h[m, k])
                assert u[m, j] == inner
                acc += int(wu[v, j]) * inner
            assert z[m, v] == acc


def test_selector_down_projection():
    # W_down = [I_r | 0] keeps the first r coordinates: z = W_up h[:, :r]
    rng = np.random.default_rng(6)
    M, d, r, V = 4, 24, 6, 40
    h = rng.standard_normal((M, d))
    wu = rng.standard_normal((V, r))
    wd = np.zeros((r, d))
    wd[np.arange(r), np.arange(r)] = 1.0
    u, z = S.lowrank_project(h, wd, wu)
    np.testing.assert_array_equal(u, h[:, :r])
    for v in range(V):
        np.testing.assert_allclose(z[:, v], (wu[v][None, :] * h[:, :r]).sum(axis=1), rtol=1e-13, atol=1e-13)


def test_identity_up_projection():
    # W_up = [I_r; 0]: the first r logits are u = W_down h, the rest are 0
    rng = np.random.default_rng(7)
    M, d, r, V = 2, 16, 5, 12
    h = rng.standard_normal((M, d))
    wd = rng.standard_normal((r, d))
    wu = np.zeros((V, r))
    wu[np.arange(r), np.arange(r)] = 1.0
    u, z = S.lowrank_project(h, wd, wu)
    for j in range(r):
        np.testing.assert_allclose(z[:, j], (wd[j][None, :] * h).sum(axis=1), rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(z[:, r:], 0.0)
    np.testing.assert_array_equal(z[:, :r], u)


def test_shapes_are_checked():
    with pytest.raises(ValueError):
        S.lowrank_project(np.zeros((2, 8)), np.zeros((8, 4)), np.zeros((10, 4)))   # W_down transposed
    with pytest.raises(ValueError):
        S.lowrank_project(np.zeros((2, 8)), np.zeros((4, 8)), np.zeros((4, 10)))   # W_up transposed


def test_lse_closed_forms_and_library():
    scipy_special = pytest.importorskip("scipy.special")
    # a constant row of V logits c: lse = c + log V exactly, every index ties -> 0
    for c, V in [(0.0, 1), (2.5, 7), (-30.0, 128256)]:
        zmax, lse, arg = S.head_stats(np.full((1, V), c))
        assert zmax[0] == c and arg[0] == 0
        assert abs(lse[0] - (c + math.log(V))) <= 1e-12 * max(1.0, abs(c))
    rng = np.random.default_rng(8)
    z = rng.standard_normal((5, 3000)) * 4.0
    zmax, lse, arg = S.head_stats(z)
    np.testing.assert_allclose(lse, scipy_special.logsumexp(z, axis=-1), rtol=0, atol=1e-12)
    assert np.all(lse >= zmax) and np.all(lse <= zmax + math.log(z.shape[1]) + 1e-12)
    # q = exp(z - lse) is a distribution
    np.testing.assert_allclose(np.exp(z - lse[:, None]).sum(axis=1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(z[np.arange(5), arg], zmax)
    # large logits do not overflow
    zmax, lse, _ = S.head_stats(np.array([[1000.0, 1000.0]]))
    assert abs(lse[0] - (1000.0 + math.log(2.0))) < 1e-12


def test_argmax_first_on_ties():
    z = np.array([[1.0, 3.0, 2.0, 3.0], [-1.0, -1.0, -2.0, -1.0]])
    _, _, arg = S.head_stats(z)
    np.testing.assert_array_equal(arg, [1, 0])


def test_mac_counts_rank_d_over_8():
    # r = d/8 with V >> d cuts the head's multiply-adds to about r/d of the full head
    d, V = 4096, 128256
    c = S.mac_counts(d, d // 8, V)
    assert c["full"] == V * d and c["lowrank"] == (d // 8) * (d + V)
    assert 0.125 < c["lowrank"] / c["full"] < 0.13
