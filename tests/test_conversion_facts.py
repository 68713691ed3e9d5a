"""The exactness facts the kernels' code conversions rest on, checked over
every input pattern in float64 (no GPU):

* every finite E4M3 code is an f16 value (the decode and prefill convert
  FP8 codes to f16 operands with no rounding);
* INT4 codes -7..7, and 16 times them (the high nibbles are read 16x), are
  f16 values;
* a bf16 row scaled by the power of two that maps its largest exponent e to
  2^14 converts to f16 exactly for every element down to 2^-28 of 2^e, and
  its largest element stays below the f16 maximum (the prefill's BF16 V rows,
  and the query rows, which take the same prescale; the kernels clamp e at
  -100, so rows whose largest value lies below 2^-100 are scaled less and
  lose their smallest elements);
* below that the conversion's error is at most half the f16 subnormal
  spacing, 2^-25 after the scaling: 2^-39 of 2^e.

The E4M3 values are built here from the format's definition (sign, 4-bit
exponent with bias 7, 3-bit mantissa, subnormals at exponent 0, S.1111.111
not a number), apart from the oracle's codec."""
import numpy as np


def _e4m3_values():
    vals = []
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e = (b >> 3) & 0xF
        m = b & 0x7
        if e == 0xF and m == 0x7:
            continue                                  # not a number
        if e == 0:
            vals.append(s * m * 2.0 ** -9)           # subnormal: m/8 x 2^-6
        else:
            vals.append(s * (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


def _exact_in_f16(x):
    x = np.asarray(x, dtype=np.float64)
    return np.array_equal(x.astype(np.float16).astype(np.float64), x)


def test_every_e4m3_code_is_an_f16_value():
    v = _e4m3_values()
    assert len(v) == 254 and np.abs(v).max() == 448.0
    assert _exact_in_f16(v)


def test_int4_codes_and_sixteen_times_them_are_f16_values():
    c = np.arange(-7, 8, dtype=np.float64)
    assert _exact_in_f16(c) and _exact_in_f16(16 * c)
    # the nibble trick: 1024 + n (n = code + 8 in 1..15) and 1024 + 16 n are f16
    # values, and subtracting the bias is exact
    n = np.arange(16, dtype=np.float64)
    assert _exact_in_f16(1024 + n) and _exact_in_f16(1024 + 16 * n)


def _finite_bf16():
    bits = np.arange(65536, dtype=np.uint32)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]         # not infinities or NaNs
    return (bits << 16).view(np.float32).astype(np.float64)


def test_bf16_row_prescale_to_f16_is_exact_down_to_2_pow_minus_28():
    x = _finite_bf16()
    x = x[x != 0]
    ex = np.floor(np.log2(np.abs(x))).astype(np.int64)
    # a row whose largest exponent is e, for every e from ex to ex + 28
    for k in range(0, 29):
        e = ex + k
        keep = e <= 127                               # a bf16 row maximum
        y = x[keep] * np.exp2(14.0 - e[keep])
        assert _exact_in_f16(y), f"{k} binades below the row maximum"
    # the row maximum itself lands in [2^14, 2^15), below the f16 maximum
    top = np.abs(x) * np.exp2(14.0 - ex)
    assert top.min() >= 2.0 ** 14 and top.max() < 2.0 ** 15 < 65504


def test_bf16_row_prescale_error_below_2_pow_minus_28_is_bounded():
    x = _finite_bf16()
    x = x[x != 0]
    ex = np.floor(np.log2(np.abs(x))).astype(np.int64)
    for k in (29, 33, 40, 60):
        e = ex + k
        keep = e <= 127
        y = x[keep] * np.exp2(14.0 - e[keep])
        got = y.astype(np.float16).astype(np.float64)
        assert np.abs(got - y).max() <= 2.0 ** -25
