"""Failure detection without a GPU fault: a bounded device-side wait that nothing
satisfies gives up, records SSD_ERR_TIMEOUT in the workspace header (read back on the
host) and the context stays usable; the same wait satisfied records nothing."""
import numpy as np
import pytest
import torch

from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    S.ssd_selftest_wait(ws, arrive=0, limit_clocks=1 << 20)        # about half a millisecond
    assert S.ssd_read_device_error(ws) == S.SSD_ERR_TIMEOUT
    assert S.ssd_read_device_error(ws) == S.SSD_OK                # read-and-clear
    S.ssd_selftest_wait(ws, arrive=1, limit_clocks=1 << 20)
    assert S.ssd_read_device_error(ws) == S.SSD_OK
    # the context still runs kernels: a small attention call afterwards is correct
    rng = np.random.default_rng(5)
    f = lambda *s: WL.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    B, NB, Dmax, Hq, Hkv, dh, P = 1, 1, 4, 4, 1, 128, 200
    t = lambda a: to_device(np.asarray(a), "cuda")
    out = S.ssd_verify_attn(t(f(B, NB * Dmax, Hq, dh)), t(f(B, Hkv, P, dh)), t(f(B, Hkv, P, dh)),
                            t(f(B, NB * Dmax, Hkv, dh)), t(f(B, NB * Dmax, Hkv, dh)), t(np.array([P], np.int32)),
                            t(np.array([[Dmax]], np.int32)), Dmax)
    torch.cuda.synchronize()
    assert torch.isfinite(out.view(torch.bfloat16).float()).all()


def test_selftest_rejects_bad_arguments():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert S.lib().ssd_selftest_wait(S._ptr(ws), 0, 0, None) == S.SSD_ERR_INVALID
    assert S.lib().ssd_selftest_wait(S._ptr(ws), 0, (1 << 32) + 1, None) == S.SSD_ERR_INVALID
    assert S.lib().ssd_selftest_wait(None, 0, 16, None) == S.SSD_ERR_WORKSPACE
