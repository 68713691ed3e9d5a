"""Pins for the oracle's prefill attention: each new token's query attends
causally (and within the window) to the cache.  The reference is torch's
float64 softmax attention on the raw inputs of a BF16 layer with an explicit
bottom-right causal (and window) mask: a library routine on independently
gathered values."""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.helpers import bf16_to_f64, bits, host_fill
from tests.test_oracle_decode import _cache, _per_seq


def _torch_prefill(q, K, V, query_start, context_lens, G, window, scale):
    """q [T, Hq, D]; K, V per sequence [L, Hkv, D] (float64)."""
    T, Hq, D = q.shape
    out = torch.zeros(T, Hq, D, dtype=torch.float64)
    for b, L in enumerate(context_lens):
        a, e = int(query_start[b]), int(query_start[b + 1])
        n = e - a
        if n == 0:
            continue
        pos = torch.arange(L - n, L)[:, None]                   # query positions
        key = torch.arange(L)[None, :]
        allowed = key <= pos
        if window > 0:
            allowed &= key > pos - window
        k = torch.from_numpy(K[b]).repeat_interleave(G, dim=1).transpose(0, 1)   # [Hq, L, D]
        v = torch.from_numpy(V[b]).repeat_interleave(G, dim=1).transpose(0, 1)
        qq = torch.from_numpy(q[a:e]).transpose(0, 1)                           # [Hq, n, D]
        s = (qq @ k.transpose(1, 2)) * scale
        s = s.masked_fill(~allowed[None], float("-inf"))
        out[a:e] = (torch.softmax(s, dim=-1) @ v).transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("window", [0, 30])
def test_bf16_prefill_equals_masked_float64_attention(window):
    w = wl.CONFIGS["tiny"]
    fill = host_fill(w)
    kc, vc, _, _ = _cache(orc.BF16, w, fill)
    # chunks of 9 and 100 tokens: the last positions of contexts 37 and 100
    qs = np.array([0, 9, 109], dtype=np.int32)
    q = bits(wl.kv_tokens(w, 109, "cpu", stream_base=700)[0][:, :1].expand(-1, w.Hq, -1)
             .contiguous())
    got = orc.prefill(orc.BF16, q, kc, vc, fill["block_table"], qs, fill["context_lens"],
                      window=window)
    K = bf16_to_f64(fill["k_bits"])
    V = bf16_to_f64(fill["v_bits"])
    starts = np.cumsum([0] + list(w.context_lens))
    Kh = [K[starts[b]:starts[b + 1]] for b in range(w.B)]
    Vh = [V[starts[b]:starts[b + 1]] for b in range(w.B)]
    ref = _torch_prefill(bf16_to_f64(q), Kh, Vh, qs, w.context_lens, w.G, window,
                         1.0 / np.sqrt(w.D))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD])
def test_quantized_prefill_equals_masked_attention_on_dequantized_cache(mode):
    w = wl.CONFIGS["tiny"]
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(mode, w, fill)
    qs = np.array([0, 37, 37 + 50], dtype=np.int32)          # whole first sequence, 50 of 100
    q = bits(wl.kv_tokens(w, 87, "cpu", stream_base=701)[1][:, :1].expand(-1, w.Hq, -1)
             .contiguous())
    got = orc.prefill(mode, q, kc, vc, fill["block_table"], qs, fill["context_lens"],
                      k_cache_scale=ks, v_cache_scale=vs, window=16)
    Kh = _per_seq(w, fill, orc.dequantize(mode, kc, ks))
    Vh = _per_seq(w, fill, orc.dequantize(mode, vc, vs))
    ref = _torch_prefill(bf16_to_f64(q), Kh, Vh, qs, w.context_lens, w.G, 16, 1.0 / np.sqrt(w.D))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_last_token_of_a_chunk_is_the_decode_of_that_token():
    w = wl.CONFIGS["tiny"]
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(orc.FP8_PER_TOKEN_HEAD, w, fill)
    qs = np.array([0, 5, 25], dtype=np.int32)
    q = bits(wl.kv_tokens(w, 25, "cpu", stream_base=702)[0][:, :1].expand(-1, w.Hq, -1)
             .contiguous())
    pre = orc.prefill(orc.FP8_PER_TOKEN_HEAD, q, kc, vc, fill["block_table"], qs,
                      fill["context_lens"], k_cache_scale=ks, v_cache_scale=vs)
    last = q[[4, 24]]
    dec = orc.decode(orc.FP8_PER_TOKEN_HEAD, last, kc, vc, fill["block_table"],
                     fill["context_lens"], k_cache_scale=ks, v_cache_scale=vs)
    assert np.array_equal(pre[[4, 24]], dec)
