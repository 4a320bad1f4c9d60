"""Pins for the oracle's BF16 conversions.

BF16 keeps the binary32 exponent and the top 7 fraction bits ("使用 Tiny-vLLM
從零開始構建高性能 LLM 推理引擎", section "Bfloat16 的選擇").  The oracle rounds
FP64 -> BF16 once, to nearest, ties to even.  These tests pin it against
torch's FP32 -> BF16 conversion (a library routine: for inputs that are exact
FP32 numbers a single rounding from FP64 must agree with it) and against hand
derived bit patterns, including a case that only a single rounding gets right.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _torch_bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_to_double_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_from_double_matches_library_on_fp32_inputs():
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties and near-ties in the 16 dropped bits
    raw[:3000] = (raw[:3000] & 0xFFFF0000) | 0x8000
    raw[3000:4000] = (raw[3000:4000] & 0xFFFF0000) | 0x7FFF
    raw[4000:5000] = (raw[4000:5000] & 0xFFFF0000) | 0x8001
    x = raw.view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle.bf16_from_f64(x.astype(np.float64))
    ref = _torch_bf16_bits_from_f32(x)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize(
    "value,bits",
    [
        (1.0, 0x3F80),
        (-2.0, 0xC000),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (1.0 + 2.0**-8, 0x3F80),                 # tie -> even (1.0)
        (1.0 + 3 * 2.0**-8, 0x3F82),             # tie -> even (1 + 2^-6)
        (1.0 + 2.0**-8 + 2.0**-40, 0x3F81),      # just above the tie: single rounding rounds up
        (float("inf"), 0x7F80),
        (-float("inf"), 0xFF80),
        (3.4e38, 0x7F80),                        # above max + half ulp -> inf
        (3.3895313892515355e38, 0x7F7F),         # largest finite BF16
        (2.0**-133, 0x0001),                     # smallest subnormal
        (1e-40, 0x0001),                         # 1.0889 * 2^-133 -> 1 quantum
        (0.4 * 2.0**-133, 0x0000),               # rounds to zero
    ],
)
def test_bf16_from_double_known_patterns(value, bits):
    assert int(oracle.bf16_from_f64(np.array([value]))[0]) == bits


def test_single_rounding_differs_from_double_rounding():
    # Via FP32 the value 1 + 2^-8 + 2^-40 first becomes the tie 1 + 2^-8 and
    # then rounds down to even; one direct rounding must go up.
    x = 1.0 + 2.0**-8 + 2.0**-40
    via_fp32 = int(_torch_bf16_bits_from_f32(np.array([x], dtype=np.float32))[0])
    direct = int(oracle.bf16_from_f64(np.array([x]))[0])
    assert via_fp32 == 0x3F80 and direct == 0x3F81
