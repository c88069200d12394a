"""The oracle's bf16 decoding and the input generator's bf16 rounding, against values
fixed by the format (bf16 is the upper 16 bits of an IEEE fp32 word) and against torch's
own bfloat16 conversion on the CPU (no GPU)."""
import numpy as np
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL


def test_bf16_decoding_of_known_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x0001, 0x7F7F, 0x7F80, 0x3EAB], np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, np.inf, 0.333984375]
    got = O.bf16_to_f64(bits)
    assert list(got) == want
    assert np.signbit(got[3])


def test_bf16_decoding_matches_torch_on_every_finite_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    with np.errstate(invalid="ignore"):          # NaN patterns
        got = O.bf16_to_f64(bits)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_generator_rounds_to_nearest_even_like_torch():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 7,
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(WL.f32_to_bf16_bits(x), ref)
