"""ssd_accept_static: the acceptance step for callers that cannot allocate device
memory (inside a stream capture, in an allocation-free serving loop, or behind
a host that owns all device memory). It runs on the library's fixed internal
scratch instead of a caller workspace; its results must equal those of
ssd_accept on the same inputs, call after call, whatever the previous call left
in that scratch, and it must not change the device's free memory. Errors its
kernels record in that scratch are read and cleared by ssd_read_static_error.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import to_device

pytestmark = pytest.mark.gpu


def _inputs(seed, B, W, Dmax, K, V, kind):
    rng = np.random.default_rng(seed)
    NB = W + 1
    blk_len = rng.integers(0, Dmax + 1, size=(B, NB)).astype(np.int32)
    blk_len[:, W] = np.where(rng.random(B) < 0.5, K, 0)
    blk_tok = rng.integers(0, V, size=(B, NB, Dmax)).astype(np.int32)
    for b in range(B):
        for k in range(NB):
            blk_tok[b, k, blk_len[b, k]:] = -1
    lg = (rng.standard_normal((B, 1 + NB * Dmax, V)) * np.sqrt(3)).astype(np.float32)
    for b in range(B):
        for k in range(NB):
            for d in range(int(rng.integers(0, blk_len[b, k] + 1))):
                r = 0 if d == 0 else 1 + k * Dmax + d - 1
                lg[b, r, blk_tok[b, k, d]] += 20.0
    dl = (rng.standard_normal((B, K, V)) * np.sqrt(3)).astype(np.float32)
    if kind == S.SSD_LOGITS_BF16:
        lg, dl = WL.f32_to_bf16_bits(lg), WL.f32_to_bf16_bits(dl)
    u_acc = WL.uniforms24(rng, (B, NB, Dmax))
    u_fin = WL.uniforms24(rng, (B,))
    dev = "cuda"
    return [to_device(a, dev) for a in (lg, dl, blk_tok, blk_len, u_acc, u_fin)]


@pytest.mark.parametrize("mode", [S.SSD_SAMPLE, S.SSD_GREEDY])
def test_static_scratch_matches_workspace_entry_point(mode):
    cases = [(11, 8, 4, 20, 5, 128256, S.SSD_LOGITS_F32),     # two different calls in a row
             (12, 3, 2, 8, 4, 151936, S.SSD_LOGITS_BF16)]
    for seed, B, W, Dmax, K, V, kind in cases:
        tgt, drf, bt, bl, ua, uf = _inputs(seed, B, W, Dmax, K, V, kind)
        ref = S.ssd_accept(tgt, drf, bt, bl, ua, uf, mode=mode, kind=kind, K=K, chain_blk=W)
        got = S.ssd_accept_static(tgt, drf, bt, bl, ua, uf, mode=mode, kind=kind, K=K, chain_blk=W)
        torch.cuda.synchronize()
        for key in ("acc_len", "best_blk", "n_out", "out_tok"):
            assert torch.equal(got[key], ref[key]), (seed, key)


def test_static_scratch_rejects_batches_beyond_its_size():
    # 2048 sequences x 101 rows x 16 chunks of partial statistics need more than 4 MiB
    B, W, Dmax, K, V = 2048, 4, 20, 0, 128256
    dev = "cuda"
    tgt = torch.zeros((1, 1, 1), device=dev)     # never read: the size check comes first
    args = S.AcceptArgs(S.SSD_GREEDY, S.SSD_LOGITS_F32, tgt.data_ptr(), None, V, tgt.data_ptr(), tgt.data_ptr(),
                        B, W, Dmax, K, -1, None, None, tgt.data_ptr(), tgt.data_ptr(), tgt.data_ptr(),
                        tgt.data_ptr(), None)
    assert S.ssd_accept_workspace_size(args) > 4 << 20
    assert S.lib().ssd_accept_static(args, None) == S.SSD_ERR_WORKSPACE


@pytest.mark.parametrize("early", [True, False])
def test_static_calls_back_to_back_and_no_allocation(early):
    """Two different calls in a row on one stream, in both row-pass modes (the second
    call's row pass starts while the first call's finish kernel may still read the
    shared array), each equal to ssd_accept; the device's free memory is the same
    before and after (checked after a first call has loaded the library's code)."""
    cases = [(21, 6, 4, 20, 5, 128256, S.SSD_LOGITS_F32), (22, 4, 4, 20, 5, 128256, S.SSD_LOGITS_F32)]
    ins = [_inputs(*c) for c in cases]
    refs, outs = [], []
    for (seed, B, W, Dmax, K, V, kind), (tgt, drf, bt, bl, ua, uf) in zip(cases, ins):
        refs.append(S.ssd_accept(tgt, drf, bt, bl, ua, uf, mode=S.SSD_SAMPLE, kind=kind, K=K, chain_blk=W))
        outs.append(S.alloc_accept_outputs(B, W + 1, Dmax, "cuda"))
    # first call on this device: the scratch address is looked up here
    S.ssd_accept_static(*ins[0], mode=S.SSD_SAMPLE, kind=cases[0][6], K=cases[0][4], chain_blk=cases[0][2],
                        out=outs[0], early_rows=early)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for rep in range(10):
        for c, x, o in zip(cases, ins, outs):
            S.ssd_accept_static(*x, mode=S.SSD_SAMPLE, kind=c[6], K=c[4], chain_blk=c[2], out=o, early_rows=early)
        torch.cuda.synchronize()
        for r, o in zip(refs, outs):
            for key in ("acc_len", "best_blk", "n_out", "out_tok"):
                assert torch.equal(o[key], r[key]), (rep, key)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert S.ssd_read_static_error() == S.SSD_OK


def test_static_error_is_read_and_cleared():
    """A device-side check that fails inside a static call (a candidate token outside
    the vocabulary) is recorded in the fixed scratch and returned once by
    ssd_read_static_error; the next read finds the word cleared."""
    S.ssd_read_static_error()                       # start from a clear word
    tgt, drf, bt, bl, ua, uf = _inputs(31, 2, 2, 8, 4, 1000, S.SSD_LOGITS_F32)
    bl[0, 0] = 3
    bt[0, 0, 0] = 1000 + 5                          # outside [0, V): checked, never read as an index
    S.ssd_accept_static(tgt, drf, bt, bl, ua, uf, mode=S.SSD_SAMPLE, kind=S.SSD_LOGITS_F32, K=4, chain_blk=2)
    assert S.ssd_read_static_error() == S.SSD_ERR_DEVICE
    assert S.ssd_read_static_error() == S.SSD_OK
