"""The fp16 V cache holds the same values as the bf16 one: checked over every
bf16 bit pattern on the host, so the claim the layout rests on (bit-identical
attention outputs for either cache) is pinned by arithmetic, not by a GPU run.

bf16 carries 8 significant bits and exponents down to 2^-126; fp16 carries 11
significant bits, normal exponents 2^-14 .. 2^15 and subnormals down to
2^-24.  So a bf16 value with magnitude in [2^-14, 65504] is an fp16 value;
smaller ones round to the nearest fp16 subnormal (ties to even, the rounding
of the conversion in both the kernel and the append), larger ones overflow."""
import numpy as np


def _all_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32)
    return (bits << np.uint32(16)).view(np.float32)


def test_normal_range_bf16_values_are_fp16_values():
    x = _all_bf16_as_f32()
    finite = np.isfinite(x)
    a = np.abs(x)
    normal = finite & (a >= 2.0 ** -14) & (a <= 65504.0)
    with np.errstate(over="ignore"):
        back = x[normal].astype(np.float16).astype(np.float32)
    assert normal.sum() == 30 * 128 * 2   # 30 fp16 binades x 128 bf16 significands x 2 signs
    np.testing.assert_array_equal(back, x[normal])


def test_tiny_values_round_to_the_nearest_fp16_subnormal():
    x = _all_bf16_as_f32()
    tiny = np.isfinite(x) & (np.abs(x) < 2.0 ** -14) & (x != 0)
    h = x[tiny].astype(np.float16).astype(np.float64)
    # the error is at most half an fp16 subnormal step, 2^-25
    assert np.max(np.abs(h - x[tiny].astype(np.float64))) <= 2.0 ** -25
    # and zero stays zero with its sign
    z = np.array([0.0, -0.0], np.float32).astype(np.float16)
    assert np.signbit(z).tolist() == [False, True]


def test_largest_exact_value_and_first_overflow():
    # 65504 is the largest fp16 value; the next bf16 value (65536) is beyond it
    assert np.float32(65504.0).astype(np.float16) == np.float16(65504.0)
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(65536.0).astype(np.float16))
