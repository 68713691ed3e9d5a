"""Pins for the oracle's FP8-query decode (the Q-scale path of "FP8 KV cache
layer skipping vs per-head scales", opening section: one Q scale per tensor
or per query head).

q_hat = E4M3(RN32(q / s)) x s, then the ordinary decode on q_hat.  The
reference here quantizes with torch's own float8_e4m3fn cast (a library
routine: round to nearest even) inside the E4M3 range, clips by hand above
it, and runs torch's float64 softmax attention on the independently
dequantized cache.
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.helpers import bf16_to_f64, bits, host_fill
from tests.test_oracle_decode import _cache, _per_seq, _torch_attention

TINY = wl.CONFIGS["tiny"]


def _torch_q_hat(q_bits, s):
    x = torch.from_numpy(bf16_to_f64(q_bits).astype(np.float32))
    y = x / torch.from_numpy(np.array(s, dtype=np.float32))[None, :, None]
    y = torch.clamp(y, -448.0, 448.0)                   # saturation (the cast would give NaN)
    v = y.to(torch.float8_e4m3fn).to(torch.float64)
    return (v * torch.from_numpy(np.array(s, dtype=np.float64))[None, :, None]).numpy()


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16])
@pytest.mark.parametrize("scales", [[0.02], [0.5], [0.004, 0.03, 0.25, 1.0]])
def test_fp8_query_decode_matches_torch_cast_and_attention(mode, scales):
    w = TINY
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(mode, w, fill)
    q = bits(wl.queries(w, "cpu"))
    s = np.broadcast_to(np.asarray(scales, dtype=np.float32), (w.Hq,))
    got = orc.decode_fp8_query(mode, q, np.asarray(scales, dtype=np.float32), kc, vc,
                               fill["block_table"], fill["context_lens"], k_cache_scale=ks,
                               v_cache_scale=vs)
    Kh = _per_seq(w, fill, orc.dequantize(mode, kc, ks))
    Vh = _per_seq(w, fill, orc.dequantize(mode, vc, vs))
    ref = _torch_attention(_torch_q_hat(q, s), Kh, Vh, fill["context_lens"], w.G)
    np.testing.assert_allclose(got.reshape(ref.shape), ref, rtol=1e-11, atol=1e-11)


def test_query_codes_round_to_even_and_saturate():
    # values on and between the E4M3 grid, and past 448
    vals = np.array([1.0, 1.0625, 1.1875, -3.25, 500.0, -1000.0, 0.0, 2.0 ** -9, 2.0 ** -10],
                    dtype=np.float32)
    q = (vals.view(np.uint32) >> 16).astype(np.uint16).reshape(1, 1, -1)
    codes, s = orc.quantize_query(q, np.array([1.0], dtype=np.float32))
    got = (codes.astype(np.uint32) << 16).view(np.float32).reshape(-1)
    want = np.array([1.0, 1.0, 1.25, -3.25, 448.0, -448.0, 0.0, 2.0 ** -9, 0.0],
                    dtype=np.float32)
    assert np.array_equal(got, want)
    assert s.tolist() == [1.0]


def test_power_of_two_scale_on_grid_values_is_the_plain_decode():
    # q already on the E4M3 grid times a power of two: quantization is exact
    w = TINY
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(orc.FP8_PER_TOKEN_HEAD, w, fill)
    q = bits(wl.queries(w, "cpu"))
    codes, _ = orc.quantize_query(q, np.array([1.0], dtype=np.float32))
    scaled = ((codes.astype(np.uint32) << 16).view(np.float32) * np.float32(0.125))
    q_on_grid = (scaled.view(np.uint32) >> 16).astype(np.uint16)
    a = orc.decode_fp8_query(orc.FP8_PER_TOKEN_HEAD, q_on_grid,
                             np.array([0.125], dtype=np.float32), kc, vc, fill["block_table"],
                             fill["context_lens"], k_cache_scale=ks, v_cache_scale=vs)
    b = orc.decode(orc.FP8_PER_TOKEN_HEAD, q_on_grid, kc, vc, fill["block_table"],
                   fill["context_lens"], k_cache_scale=ks, v_cache_scale=vs)
    np.testing.assert_allclose(a.reshape(b.shape), b, rtol=1e-13, atol=1e-13)
