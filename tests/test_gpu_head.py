"""GPU parity of the low-rank draft head (SlimSpec page, "방법론: SlimSpec" / "아키텍처":
z = W_up W_down h; q = softmax(z)) through the C ABI, against the fp64 oracle.

Tolerance, from the kernel's arithmetic: u = W_down h is accumulated in fp32 and
rounded to bf16 (relative error <= 2^-9, and an fp32 error in u can move the
rounding by one more bf16 step, so 2^-8 covers both); z = W_up u is accumulated
in fp32. Per logit:
    |z_gpu - z| <= sum_j |W_up[v,j]| (2^-8 |u_j| + 2^-16 A_j) + 2^-16 sum_j |W_up[v,j] u_j| + 1e-6,
with A_j = sum_k |W_down[j,k] h_k| (fp32 accumulation of d products, taken with
a few times the typical sqrt(d) 2^-24 random-walk size). A second, tighter check
models the bf16 rounding on the oracle's own u.
"""
import math

import numpy as np
import pytest
import torch

from oracle import slimspec_oracle as S
from oracle.ssd_oracle import bf16_to_f64
from speculative_decoding_copy_gb300 import _binding as ssd
from speculative_decoding_copy_gb300.workloads import (HEAD_WORKLOADS, HeadWorkload, bf16_bits_to_f32,
                                                       f32_to_bf16_bits, make_head_inputs)

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)


def _bound(x, o):
    h, wd, wu = bf16_to_f64(x["h"]), bf16_to_f64(x["w_down"]), bf16_to_f64(x["w_up"])
    A = np.abs(h) @ np.abs(wd).T                      # [M][r]
    au = np.abs(o["u"])
    awu = np.abs(wu)
    return (2.0 ** -8 * au + 2.0 ** -16 * A) @ awu.T + 2.0 ** -16 * (au @ awu.T) + 1e-6


def _run(x, logits_dtype=torch.float32):
    h, wd, wu = _dev(x["h"]), _dev(x["w_down"]), _dev(x["w_up"])
    row_max, lse, arg, logits, ws = ssd.ssd_lowrank_head(h, wd, wu, logits_dtype=logits_dtype)
    torch.cuda.synchronize()
    assert ssd.ssd_read_device_error(ws) == 0
    return (row_max.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            arg.cpu().numpy().astype(np.int64),
            None if logits is None else logits.float().cpu().numpy().astype(np.float64))


def _check(x, logits_dtype=torch.float32):
    o = S.slimspec_head(x["h"], x["w_down"], x["w_up"])
    bound = _bound(x, o)
    row_max, lse, arg, z = _run(x, logits_dtype)
    M, V = o["z"].shape
    tol_row = bound.max(axis=1)
    if z is not None:
        err = np.abs(z - o["z"])
        if logits_dtype == torch.bfloat16:
            err_ok = err <= bound + 2.0 ** -8 * np.abs(o["z"])       # plus the output rounding
        else:
            err_ok = err <= bound
        assert err_ok.all(), f"{(~err_ok).sum()} logits out of bound; worst excess {(err - bound).max()}"
        if logits_dtype == torch.float32:
            # tighter: the oracle's u rounded to bf16, then the exact second product
            ub = bf16_to_f64(f32_to_bf16_bits(o["u"].astype(np.float32)))
            zt = ub @ bf16_to_f64(x["w_up"]).T
            aw = np.abs(bf16_to_f64(x["w_up"]))
            tight = 4 * 2.0 ** -8 * aw.max(axis=1)[None, :] * np.abs(o["u"]).max(axis=1)[:, None] + \
                2.0 ** -14 * (np.abs(ub) @ aw.T) + 1e-6
            assert (np.abs(z - zt) <= tight).all()
            # the statistics agree exactly with the kernel's own logits
            np.testing.assert_array_equal(row_max, z.max(axis=1))
            np.testing.assert_array_equal(arg, np.argmax(z, axis=1))
            lse_own = z.max(axis=1) + np.log(np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1))
            lerr = np.abs(lse - lse_own)
            assert (lerr <= 2e-5 * np.maximum(1.0, np.abs(lse_own))).all(), f"lse vs own logits: {lerr.max()}"
    # against the oracle
    assert (np.abs(row_max - o["row_max"]) <= tol_row).all()
    assert (np.abs(lse - o["lse"]) <= tol_row + 2e-5 * np.maximum(1.0, np.abs(o["lse"]))).all()
    assert ((arg >= 0) & (arg < V)).all()
    assert (o["z"][np.arange(M), arg] >= o["row_max"] - 2 * tol_row).all()
    return o, (row_max, lse, arg, z)


def test_small_workload():
    _check(make_head_inputs(HEAD_WORKLOADS["head_small"]))


@pytest.mark.parametrize("M,d,r,V", [
    (1, 64, 64, 128),          # one tile, one atom each
    (16, 520, 200, 1),         # a single logit; d and r not multiples of 64
    (17, 8, 8, 129),           # the smallest d and r; one row in the second tile
    (33, 1024, 128, 5000),     # two column groups
    (64, 2048, 1024, 3001),    # the largest batch and rank
    (48, 4096, 512, 20000),    # N = 48, a full-size hidden state
])
def test_shapes(M, d, r, V):
    hw = HeadWorkload(f"t{M}_{d}_{r}_{V}", M=M, d=d, r=r, V=V, z_std=3.0)
    _check(make_head_inputs(hw, seed=1000 + M + d + r + V))


def test_bf16_logits():
    _check(make_head_inputs(HEAD_WORKLOADS["head_small"], seed=77), logits_dtype=torch.bfloat16)


def test_stats_only():
    x = make_head_inputs(HeadWorkload("s", M=9, d=256, r=64, V=3000, z_std=3.0), seed=78)
    _check(x, logits_dtype=None)


@pytest.mark.parametrize("name", ["head_llama8b_b64", "head_llama8b_b1"])
def test_full_size(name):
    _check(make_head_inputs(HEAD_WORKLOADS[name]))


def test_ties_take_the_lowest_index():
    # rows 7, 300 and 9000 of W_up are the same large row: equal logits, the max of every batch row
    hw = HeadWorkload("ties", M=4, d=256, r=64, V=10000, z_std=1.0)
    x = make_head_inputs(hw, seed=79)
    wu = bf16_bits_to_f32(x["w_up"]).copy()
    o = S.slimspec_head(x["h"], x["w_down"], x["w_up"])
    sign = np.sign(o["u"].sum(axis=0))          # a row aligned with the batch's u
    big = (sign * 0.5).astype(np.float32)
    for v in (9000, 300, 7):
        wu[v] = big
    x["w_up"] = f32_to_bf16_bits(wu)
    o = S.slimspec_head(x["h"], x["w_down"], x["w_up"])
    assert (o["argmax"] == 7).all()
    _, (_, _, arg, z) = _check(x)
    np.testing.assert_array_equal(arg, 7)
    np.testing.assert_array_equal(z[:, 7], z[:, 300])


def test_repeat_calls_are_identical():
    x = make_head_inputs(HeadWorkload("rep", M=20, d=1024, r=256, V=7000, z_std=3.0), seed=80)
    a = _run(x)
    b = _run(x)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_invalid_arguments_launch_nothing():
    dev = torch.device("cuda")
    h = torch.zeros(65, 64, dtype=torch.bfloat16, device=dev)
    wd = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    wu = torch.zeros(100, 64, dtype=torch.bfloat16, device=dev)
    before = ssd.launch_count()
    with pytest.raises(ssd.SsdError):
        ssd.ssd_lowrank_head(h, wd, wu)                 # M = 65
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_lowrank_head(h[:4], torch.zeros(1032, 64, dtype=torch.bfloat16, device=dev),
                             torch.zeros(100, 1032, dtype=torch.bfloat16, device=dev))   # r > 1024
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_lowrank_head(h[:4, :60].contiguous(), wd[:, :60].contiguous(), wu)      # d = 60, not a multiple of 8
    assert e.value.status in (ssd.SSD_ERR_UNSUPPORTED, ssd.SSD_ERR_INVALID)
    assert ssd.launch_count() == before
