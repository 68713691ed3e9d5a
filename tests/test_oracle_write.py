"""Pins for the oracle's cache write.

Rules: scale = amax/448 (FP8) or amax/7 (INT4), 1.0 when amax is 0, one FP32
scale per token-head slot ("Per-tensor vs per-head FP8 KV cache scales",
section "Dynamic per-token-head scales add 3.125 percent"; "Per-token-head KV
cache scale overhead", section "INT4 makes the metadata fraction larger");
per-tensor and static per-head scales come from the caller (same page,
section "Per-tensor vs per-head FP8 KV cache scales").
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.helpers import bf16_to_f64, bits, from_bits, host_fill

TINY = wl.CONFIGS["tiny"]


def _write(mode, w, fill, k_scale=None, v_scale=None):
    pg = fill["paging"]
    kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, w.Hkv, w.block_size, w.D)
    orc.cache_write(mode, fill["k_bits"], fill["v_bits"], fill["slots_np"], kc, vc, ks, vs,
                    k_scale=k_scale, v_scale=v_scale, block_size=w.block_size)
    return kc, vc, ks, vs


def _gather_rows(w, fill, cache):
    """Cache rows in token order (token t lives at slot slots[t])."""
    s = fill["slots_np"]
    blk, off = s // w.block_size, s % w.block_size
    return cache[blk, :, off]            # [T, Hkv, row]


def test_dynamic_fp8_amax_maps_to_448_and_scale_is_fp32_quotient():
    fill = host_fill(TINY)
    kc, vc, ks, vs = _write(orc.FP8_PER_TOKEN_HEAD, TINY, fill)
    table = orc.e4m3_decode_table()
    for codes, scales, x in ((kc, ks, fill["k_bits"]), (vc, vs, fill["v_bits"])):
        rows = _gather_rows(TINY, fill, codes)
        sc = scales[fill["slots_np"] // 16, :, fill["slots_np"] % 16]
        amax = np.abs(bf16_to_f64(x)).max(axis=-1).astype(np.float32)
        expect = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0))
        assert np.array_equal(sc, expect)
        mags = np.abs(table[rows]).max(axis=-1)
        assert np.all(mags == 448.0)
        # the element holding the amax is the one that maps to +-448
        arg = np.abs(bf16_to_f64(x)).argmax(axis=-1)
        picked = np.take_along_axis(rows, arg[..., None], axis=-1)[..., 0]
        assert np.all((picked & 0x7F) == 0x7E)


def test_dynamic_int4_amax_maps_to_7():
    fill = host_fill(TINY)
    kc, vc, ks, vs = _write(orc.INT4_PER_TOKEN_HEAD, TINY, fill)
    s = fill["slots_np"]
    deq = orc.dequantize(orc.INT4_PER_TOKEN_HEAD, kc, ks)[s // 16, :, s % 16]
    used = deq / ks[s // 16, :, s % 16][..., None].astype(np.float64)
    assert np.all(np.abs(used).max(axis=-1) == 7.0)
    assert np.all(used == np.round(used)) and np.all(np.abs(used) <= 7)


def test_zero_vector_gets_scale_one_and_zero_codes():
    T, Hkv, D = 3, 2, 64
    x = np.zeros((T, Hkv, D), dtype=np.uint16)
    x[1, 1, 5] = 0x8000   # -0.0 keeps its sign bit
    slots = np.array([0, 17, 33], dtype=np.int64)
    for mode in (orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD):
        kc, vc, ks, vs = orc.alloc_cache(mode, 3, Hkv, 16, D)
        orc.cache_write(mode, x, x, slots, kc, vc, ks, vs)
        assert np.all(ks[slots // 16, :, slots % 16] == 1.0)
        if mode == orc.FP8_PER_TOKEN_HEAD:
            assert kc[1, 1, 1, 5] == 0x80
            kc[1, 1, 1, 5] = 0
        assert not kc.any()


def test_negative_slots_leave_cache_untouched():
    fill = host_fill(TINY)
    slots = fill["slots_np"].copy()
    skip = np.arange(len(slots)) % 3 == 0
    slots[skip] = -1
    pg = fill["paging"]
    for mode in range(5):
        kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, 2, 16, 64)
        kc[:] = 0xA5
        if ks is not None:
            ks[:] = -3.0
        sc = np.array([0.5, 2.0], dtype=np.float32)
        orc.cache_write(mode, fill["k_bits"], fill["v_bits"], slots, kc, vc, ks, vs,
                        k_scale=sc, v_scale=sc)
        s = fill["slots_np"][skip]
        assert np.all(kc[s // 16, :, s % 16] == 0xA5)
        if ks is not None:
            assert np.all(ks[s // 16, :, s % 16] == -3.0)


def test_slot_outside_cache_is_an_error():
    x = np.zeros((1, 2, 64), dtype=np.uint16)
    kc, vc, ks, vs = orc.alloc_cache(orc.FP8_PER_TOKEN_HEAD, 2, 2, 16, 64)
    with pytest.raises(ValueError):
        orc.cache_write(orc.FP8_PER_TOKEN_HEAD, x, x, np.array([32]), kc, vc, ks, vs)


def test_per_tensor_scale_one_on_representable_inputs_is_a_plain_cast():
    # Inputs that are exactly E4M3 values: a per-tensor scale of 1.0 must give
    # torch's float8_e4m3fn cast, scattered to the right slots.
    w = TINY
    fill = host_fill(w)
    T = fill["T"]
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    codes = rng.choice(finite, size=(T, w.Hkv, w.D)).astype(np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.bfloat16)
    xb = bits(vals)
    one = np.ones(1, dtype=np.float32)
    fill = dict(fill, k_bits=xb, v_bits=xb)
    kc, vc, _, _ = _write(orc.FP8_PER_TENSOR, w, fill, k_scale=one, v_scale=one)
    ref = vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(_gather_rows(w, fill, kc), ref)
    assert np.array_equal(_gather_rows(w, fill, vc), ref)


def test_bf16_layer_is_a_byte_copy_to_the_slot():
    fill = host_fill(TINY)
    kc, vc, ks, vs = _write(orc.BF16, TINY, fill)
    assert ks is None
    rows = _gather_rows(TINY, fill, kc).view(np.uint16)
    assert np.array_equal(rows, fill["k_bits"])


def test_closed_form_error_bounds():
    # FP8 RNE: relative error <= 2^-4 for normals, absolute <= 2^-10 * s in the
    # subnormal range; the fp32 division adds <= 2^-24 relative.  INT4: <= s/2.
    fill = host_fill(TINY)
    x = bf16_to_f64(fill["k_bits"])
    s = fill["slots_np"]
    kc, vc, ks, vs = _write(orc.FP8_PER_TOKEN_HEAD, TINY, fill)
    xh = orc.dequantize(orc.FP8_PER_TOKEN_HEAD, kc, ks)[s // 16, :, s % 16]
    sc = ks[s // 16, :, s % 16][..., None].astype(np.float64)
    bound = sc * np.maximum(2.0 ** -4 * np.abs(x / sc), 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(np.abs(x - xh) <= bound)
    kc, vc, ks, vs = _write(orc.INT4_PER_TOKEN_HEAD, TINY, fill)
    xh = orc.dequantize(orc.INT4_PER_TOKEN_HEAD, kc, ks)[s // 16, :, s % 16]
    sc = ks[s // 16, :, s % 16][..., None].astype(np.float64)
    assert np.all(np.abs(x - xh) <= sc * 0.5 * (1 + 2.0 ** -20))


def test_range_sharing_error_ordering():
    # One scale shared across heads spends range on the big head; finer scales
    # lower the error of small heads ("Range sharing explains the accuracy
    # trade").  Mean relative error: dynamic <= static per-head <= per-tensor.
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=2, context=256)
    fill = host_fill(w)
    x = bf16_to_f64(fill["k_bits"])
    s = fill["slots_np"]
    cal_k, _ = wl.calibration_sample(w, "cpu")
    head = orc.calibrate_per_head(bits(cal_k))
    tensor = np.array([head.max()], dtype=np.float32)
    errs = {}
    for mode, sc in ((orc.FP8_PER_TENSOR, tensor), (orc.FP8_PER_HEAD, head),
                     (orc.FP8_PER_TOKEN_HEAD, None)):
        kc, vc, ks, vs = _write(mode, w, fill, k_scale=sc, v_scale=sc)
        xh = orc.dequantize(mode, kc, ks, sc)[s // 16, :, s % 16]
        errs[mode] = float(np.mean(np.abs(x - xh) / (np.abs(x) + 1e-3)))
    assert errs[orc.FP8_PER_TOKEN_HEAD] <= errs[orc.FP8_PER_HEAD] <= errs[orc.FP8_PER_TENSOR]


def test_range_sharing_example_one_sixteenth():
    # A head at 32 and a head at 2 under one shared scale: the small head spans
    # 1/16 of the represented range.
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "accounting.json")))
    r = g["range_sharing"]
    shared = max(r["large_head_amax"], r["small_head_amax"]) / 448.0
    x = np.zeros((1, 2, 64), dtype=np.uint16)
    vals = torch.zeros(1, 2, 64)
    vals[0, 0, 0] = r["large_head_amax"]
    vals[0, 1, 0] = r["small_head_amax"]
    xb = bits(vals.to(torch.bfloat16))
    kc, vc, _, _ = orc.alloc_cache(orc.FP8_PER_TENSOR, 1, 2, 16, 64)
    sc = np.array([shared], dtype=np.float32)
    orc.cache_write(orc.FP8_PER_TENSOR, xb, xb, np.array([0]), kc, vc, None, None,
                    k_scale=sc, v_scale=sc)
    table = orc.e4m3_decode_table()
    assert table[kc[0, 1, 0, 0]] / table[kc[0, 0, 0, 0]] == r["fraction_of_range"]


def test_calibration_is_per_head_amax_over_448():
    w = wl.CONFIGS["llama8b"]
    k, _ = wl.calibration_sample(w, "cpu")
    xb = bits(k)
    got = orc.calibrate_per_head(xb)
    amax = np.abs(bf16_to_f64(xb)).max(axis=(0, 2)).astype(np.float32)
    assert np.array_equal(got, amax / np.float32(448.0))


def _one_vector(mode, values, D=64):
    """Writes one token (one KV head) whose first elements are `values` (the
    rest zero) to slot 0 and returns its code row and scale."""
    x = torch.zeros((1, 1, D), dtype=torch.bfloat16)
    x[0, 0, :len(values)] = torch.tensor(values, dtype=torch.float64).to(torch.bfloat16)
    xb = bits(x)
    kc, vc, ks, vs = orc.alloc_cache(mode, 1, 1, 16, D)
    orc.cache_write(mode, xb, xb, np.zeros(1, dtype=np.int64), kc, vc, ks, vs)
    assert np.array_equal(kc, vc) and np.array_equal(ks, vs)
    return kc[0, 0, 0], ks[0, 0, 0]


def test_int4_packing_hand_computed_bytes():
    """Packed INT4 ("Per-token-head KV cache scale overhead", section "INT4
    makes the metadata fraction larger": widths halved, two values a byte),
    read as two's-complement nibbles with the even element in the low
    nibble.  The bytes below are worked out by hand, not by the oracle."""
    # amax 7 -> scale 1: the codes are the values themselves, -7..7 then -7
    row, s = _one_vector(orc.INT4_PER_TOKEN_HEAD,
                         [-7, -6, -5, -4, -3, -2, -1, 0, 1, 2, 3, 4, 5, 6, 7, -7])
    assert s == 1.0
    assert list(row[:8]) == [0xA9, 0xCB, 0xED, 0x0F, 0x21, 0x43, 0x65, 0x97]
    assert not row[8:].any()
    # amax 14 -> scale 2: 14/2 = 7, -3/2 = -1.5 -> -2, 5/2 = 2.5 -> 2 (ties to
    # even), 1/2 = 0.5 -> 0, -13/2 = -6.5 -> -6, 9/2 = 4.5 -> 4
    row, s = _one_vector(orc.INT4_PER_TOKEN_HEAD, [14, -3, 5, 1, -13, 9])
    assert s == 2.0
    assert list(row[:3]) == [0xE7, 0x02, 0x4A]
    assert not row[3:].any()


def test_fp8_dynamic_hand_computed_codes():
    """Dynamic FP8: scale = amax/448 in fp32, codes are E4M3 of x/scale
    ("Per-tensor vs per-head FP8 KV cache scales", section "Dynamic
    per-token-head scales add 3.125 percent").  amax 448 gives scale 1, so
    the codes are the E4M3 encodings of the values, worked out by hand:
    448 = 1.75 x 2^8 -> 0x7E; -224 = -1.75 x 2^7 -> 0xF6; 1 -> 0x38;
    0.3125 = 1.25 x 2^-2 -> 0x2A; 2^-9 (smallest subnormal) -> 0x01;
    -17 lies halfway between -16 and -18 (spacing 2 at 2^4) and takes the even
    mantissa, -16 = -1.0 x 2^4 -> 0xD8."""
    row, s = _one_vector(orc.FP8_PER_TOKEN_HEAD, [448, -224, 1, 0.3125, 2.0 ** -9, -17])
    assert s == 1.0
    assert list(row[:6]) == [0x7E, 0xF6, 0x38, 0x2A, 0x01, 0xD8]
    assert not row[6:].any()


def _static_write(mode, k_scale, v_scale, values, D=64):
    """One token, two KV heads, both heads' K and V holding `values` (then
    zeros), written with distinct K and V scales; returns the K and V code
    rows [2, D]."""
    x = torch.zeros((1, 2, D), dtype=torch.bfloat16)
    x[0, :, :len(values)] = torch.tensor(values, dtype=torch.float64).to(torch.bfloat16)
    xb = bits(x)
    kc, vc, _, _ = orc.alloc_cache(mode, 1, 2, 16, D)
    orc.cache_write(mode, xb, xb, np.zeros(1, dtype=np.int64), kc, vc, None, None,
                    k_scale=np.asarray(k_scale, dtype=np.float32),
                    v_scale=np.asarray(v_scale, dtype=np.float32))
    return kc[0, :, 0], vc[0, :, 0]


# E4M3 codes worked out by hand (bias 7; code = sign | E << 3 | M, value
# 2^(E-7) (1 + M/8)) for the quotients y = x / s of x = 1, -3, 100, 300:
#   y = 2 -> 0x40, -6 -> 0xCC, 200 (halfway 192|208, even M) -> 0x74, 600 -> 0x7E (saturated)
#   y = 0.25 -> 0x28, -0.75 -> 0xB4, 25 (halfway 24|26) -> 0x5C, 75 (-> 72) -> 0x69
#   y = 0.5 -> 0x30, -1.5 -> 0xBC, 50 (halfway 48|52) -> 0x64, 150 (-> 144) -> 0x71
#   y = 4 -> 0x48, -12 -> 0xD4, 400 (halfway 384|416) -> 0x7C, 1200 -> 0x7E
HAND = {0.5: [0x40, 0xCC, 0x74, 0x7E], 4.0: [0x28, 0xB4, 0x5C, 0x69],
        2.0: [0x30, 0xBC, 0x64, 0x71], 0.25: [0x48, 0xD4, 0x7C, 0x7E]}
VALUES = [1, -3, 100, 300]


def test_static_per_head_distinct_k_and_v_scales_hand_computed():
    """Static per-head FP8 ("Per-tensor vs per-head FP8 KV cache scales",
    section "Static per-head metadata is almost free": one K and one V scale
    per KV head): head h of K divides by k_scale[h], head h of V by
    v_scale[h].  Four distinct scales, so a K/V or a head swap changes bytes."""
    kc, vc = _static_write(orc.FP8_PER_HEAD, [0.5, 4.0], [2.0, 0.25], VALUES)
    assert list(kc[0, :4]) == HAND[0.5] and list(kc[1, :4]) == HAND[4.0]
    assert list(vc[0, :4]) == HAND[2.0] and list(vc[1, :4]) == HAND[0.25]
    assert not kc[:, 4:].any() and not vc[:, 4:].any()


def test_per_tensor_distinct_k_and_v_scales_hand_computed():
    """Per-tensor FP8 (same page and section: one K and one V scale per
    layer): every head of K divides by k_scale[0], every head of V by
    v_scale[0]."""
    kc, vc = _static_write(orc.FP8_PER_TENSOR, [0.5], [2.0], VALUES)
    assert list(kc[0, :4]) == HAND[0.5] and list(kc[1, :4]) == HAND[0.5]
    assert list(vc[0, :4]) == HAND[2.0] and list(vc[1, :4]) == HAND[2.0]
