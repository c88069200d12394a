"""Host-side logic of the step driver (no GPU): the input arena that lets a caller
refresh every input of a step with one host-to-device copy."""
import numpy as np
import pytest
import torch

from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import ARENA_ALIGN, VerifyStep, arena_bytes, default_early_rows


@pytest.mark.parametrize("with_attention", [True, False])
def test_arena_views_are_aligned_disjoint_and_hold_the_inputs(with_attention):
    wl = WL.WORKLOADS["tiny"]
    inp = WL.make_inputs(wl, 5, full_width=False)
    n = arena_bytes(inp, with_attention)
    arena = torch.zeros(n, dtype=torch.uint8)
    st = VerifyStep(wl, inp, device="cpu", arena=arena, with_attention=with_attention)
    ref = VerifyStep(wl, inp, device="cpu", with_attention=with_attention)
    assert set(st.x) == set(ref.x)
    spans = []
    for k, t in st.x.items():
        off = t.data_ptr() - arena.data_ptr()
        assert off % ARENA_ALIGN == 0, k
        assert t.is_contiguous() and 0 <= off and off + t.numel() * t.element_size() <= n, k
        spans.append((off, off + t.numel() * t.element_size()))
        assert t.dtype == ref.x[k].dtype and t.shape == ref.x[k].shape, k
        assert torch.equal(t, ref.x[k]), k
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    # one copy of a same-layout buffer refreshes every input
    other = WL.make_inputs(wl, 6, full_width=False)
    src = torch.zeros(n, dtype=torch.uint8)
    VerifyStep(wl, other, device="cpu", arena=src, with_attention=with_attention)
    arena.copy_(src)
    again = VerifyStep(wl, other, device="cpu", with_attention=with_attention)
    for k, t in st.x.items():
        assert torch.equal(t, again.x[k]), k


def test_arena_too_small_is_rejected():
    wl = WL.WORKLOADS["tiny"]
    inp = WL.make_inputs(wl, 5, full_width=False)
    with pytest.raises(ValueError):
        VerifyStep(wl, inp, device="cpu", arena=torch.zeros(arena_bytes(inp) - 1, dtype=torch.uint8))
    with pytest.raises(ValueError):
        VerifyStep(wl, inp, device="cpu", order="sideways")


def test_step_defaults_per_workload():
    """Early row pass where every row is needed anyway; tile skipping in the attention only
    for batches whose gate can send sequences to the chain draft."""
    W = WL.WORKLOADS
    assert default_early_rows(W["llama8b"]) and default_early_rows(W["llama70b"])
    assert not default_early_rows(W["batched"]) and not default_early_rows(W["qwen8b_mixed"])
    inp = WL.make_inputs(W["tiny"], 5, full_width=False)
    assert VerifyStep(W["tiny"], inp, device="cpu").skip_absent is False          # a single sequence
    assert VerifyStep(W["tiny"], inp, device="cpu", skip_absent=True).skip_absent is True
