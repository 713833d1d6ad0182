"""Pins for the oracle's float64 -> bf16 rounding (round to nearest even).

Checked against torch's fp32 -> bf16 conversion (a library routine) on fp32
inputs, and against hand-worked values where a float64 differs from every
fp32 (a rounding taken through fp32 first would round twice)."""
import math

import numpy as np
import pytest
import torch

import oracle


def _torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),   # fp32 subnormals
        (rng.standard_normal(5000) * 1e-40).astype(np.float32),
        # exact halfway points between neighbouring bf16 values
        ((rng.integers(0, 1 << 15, 5000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, -3.3895314e38], dtype=np.float32),
    ]
    v = np.concatenate(parts)
    v = v[np.isfinite(v)]
    got = oracle.f64_to_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, _torch_bf16_bits(v))


@pytest.mark.parametrize("value, expected", [
    (1.0 + 2.0 ** -8, 1.0),                       # halfway, even neighbour is 1.0
    (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),       # halfway, even neighbour above
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -7),  # just above halfway (fp32 would make it a tie)
    (1.0 + 2.0 ** -8 - 2.0 ** -40, 1.0),          # just below halfway
    (-(1.0 + 2.0 ** -8 + 2.0 ** -30), -(1.0 + 2.0 ** -7)),
    (2.0 ** -133, 2.0 ** -133),                   # smallest bf16 subnormal
    (2.0 ** -134, 0.0),                           # halfway to zero: ties to even (zero)
    (1.5 * 2.0 ** -134, 2.0 ** -133),
    ((2 - 2.0 ** -7) * 2.0 ** 127, (2 - 2.0 ** -7) * 2.0 ** 127),  # largest finite bf16
    ((2 - 2.0 ** -8) * 2.0 ** 127, math.inf),     # halfway to the next binade: overflow
])
def test_direct_rounding_cases(value, expected):
    got = oracle.f64_to_bf16(np.array([value]))
    ref = np.array([expected], dtype=np.float32).view(np.uint32) >> 16
    assert int(got[0]) == int(ref[0]), (value, hex(int(got[0])), hex(int(ref[0])))


def test_signed_zero_and_nan():
    got = oracle.f64_to_bf16(np.array([0.0, -0.0, math.nan, math.inf, -math.inf]))
    assert list(got[:2]) == [0x0000, 0x8000]
    assert (got[2] & 0x7F80) == 0x7F80 and (got[2] & 0x7F) != 0
    assert list(got[3:]) == [0x7F80, 0xFF80]


def test_roundtrip_of_bf16_values_is_identity():
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]  # finite only
    np.testing.assert_array_equal(oracle.f64_to_bf16(oracle.bf16_to_f64(b)), b)
