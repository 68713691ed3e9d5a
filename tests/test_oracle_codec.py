"""Pins for the oracle's E4M3 and INT4 codecs.

The E4M3 format is the OCP "fn" variant (max 448, no infinities); the pages
only say that values outside the chosen range clip ("Per-tensor vs per-head
FP8 KV cache scales", section "Range sharing explains the accuracy trade").
Pins: torch's float8_e4m3fn decode of all 256 codes, torch's cast for
in-range values, a brute-force nearest-value search, round trips and
saturation.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_float8_for_all_256_codes():
    ours = orc.e4m3_decode_table()
    ref = _torch_decode_all()
    nan_ours = np.isnan(ours)
    assert list(np.nonzero(nan_ours)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ref), nan_ours)
    assert np.array_equal(ours[~nan_ours], ref[~nan_ours])
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_round_trip_every_finite_code():
    table = orc.e4m3_decode_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(np.float32(table[c])) == c, hex(c)


def _nearest_even_by_search(y, table):
    """Brute force: the finite code nearest to y; ties go to the even code."""
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    best = None
    for c in finite:
        d = abs(table[c] - y)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1)):
            best = (d, c)
    return best[1]


def test_encode_matches_brute_force_nearest_search():
    table = orc.e4m3_decode_table()
    rng = np.random.default_rng(7)
    exps = rng.uniform(-12, 8.8, size=600)
    ys = (np.sign(rng.standard_normal(600)) * 2.0 ** exps).astype(np.float32)
    # exact midpoints between neighbouring positive codes, and one fp32 ulp around them
    pos = sorted(table[c] for c in range(0x7F))
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    extra = []
    for m in mids:
        f = np.float32(m)
        extra += [f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(1e9))]
    for y in list(ys) + extra + [-np.float32(m) for m in mids]:
        if abs(float(y)) >= 448:
            continue
        ref = _nearest_even_by_search(float(y), table)
        got = orc.e4m3_encode(y)
        # -0 and +0 are both "nearest" to a tiny value: the encoder keeps the sign
        if table[ref] == 0.0:
            assert got in (0x00, 0x80) and (got >> 7) == (1 if np.signbit(y) else 0), y
        else:
            assert got == ref, (float(y), hex(got), hex(ref))


def test_encode_matches_torch_cast_on_all_in_range_bf16_values():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = bits.float()
    keep = torch.isfinite(vals) & (vals.abs() < 448)
    vals = vals[keep]
    ref = vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(v) for v in vals.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_saturation_and_specials():
    assert orc.e4m3_encode(448.0) == 0x7E
    assert orc.e4m3_encode(463.9) == 0x7E
    assert orc.e4m3_encode(464.0) == 0x7E
    assert orc.e4m3_encode(1e30) == 0x7E
    assert orc.e4m3_encode(float("inf")) == 0x7E
    assert orc.e4m3_encode(-float("inf")) == 0xFE
    assert orc.e4m3_encode(-500.0) == 0xFE
    assert orc.e4m3_encode(float("nan")) & 0x7F == 0x7F
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(-1e-30) == 0x80
    # half of the smallest subnormal is a tie between 0 and 2^-9: even -> 0
    assert orc.e4m3_encode(2.0 ** -10) == 0x00
    assert orc.e4m3_encode(3 * 2.0 ** -10) == 0x02      # tie 1.5 -> 2
    # top of the subnormal range rounds up into the first normal
    assert orc.e4m3_encode(7.75 * 2.0 ** -9) == 0x08
    # mantissa carry into the exponent: 15.5 lies halfway between 15 and 16
    assert orc.e4m3_encode(15.5) == orc.e4m3_encode(16.0)


def test_int4_round_half_even_and_clamp():
    ys = np.linspace(-9.0, 9.0, 7201, dtype=np.float32)
    got = np.array([orc.int4_encode(y) for y in ys])
    ref = np.clip(np.round(ys), -7, 7).astype(int)   # numpy rounds half to even
    assert np.array_equal(got, ref)
    assert [orc.int4_encode(v) for v in (0.5, 1.5, 2.5, -2.5, 6.5, 7.4999)] == [0, 2, 2, -2, 6, 7]


def test_array_encoder_matches_scalar_encoder():
    rng = np.random.default_rng(11)
    y = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    out = np.empty(y.size, dtype=np.uint8)
    orc.lib().orc_e4m3_encode_array(y.ctypes.data, out.ctypes.data, y.size)
    ref = np.array([orc.e4m3_encode(v) for v in y], dtype=np.uint8)
    assert np.array_equal(out, ref)
