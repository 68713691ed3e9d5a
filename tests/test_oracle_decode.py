"""Pins for the oracle's paged decode attention.

Definition: out[b, hq] = sum_p softmax_p(scale * <q[b,hq], K_hat[p, hq // G]>) V_hat[p]
over retained positions p in [lo, L), lo = max(0, L - W) for a window W
("FP8 KV cache layer skipping vs per-head scales", section "Layer skipping
follows retained-token footprint"), on the dequantized cache.  Pins: torch's
float64 softmax/matmul on independently dequantized values, L = 1, K = 0,
W >= L, the window as a slice, and the GQA head grouping.
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.helpers import bf16_to_f64, bits, host_fill

TINY = wl.CONFIGS["tiny"]


def _cache(mode, w, fill, sc=None):
    pg = fill["paging"]
    kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, w.Hkv, w.block_size, w.D)
    orc.cache_write(mode, fill["k_bits"], fill["v_bits"], fill["slots_np"], kc, vc, ks, vs,
                    k_scale=sc, v_scale=sc, block_size=w.block_size)
    return kc, vc, ks, vs


def _torch_attention(q, Kh, Vh, context_lens, G, window=0, scale=None):
    """Library reference: per sequence, float64 softmax(q K^T * scale) V."""
    B, Hq, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        L = int(context_lens[b])
        lo = max(0, L - window) if window > 0 else 0
        if L <= lo:
            continue
        k = torch.from_numpy(Kh[b][lo:L])   # [n, Hkv, D]
        v = torch.from_numpy(Vh[b][lo:L])
        k = k.repeat_interleave(G, dim=1).transpose(0, 1)   # [Hq, n, D]
        v = v.repeat_interleave(G, dim=1).transpose(0, 1)
        qq = torch.from_numpy(q[b])[:, None, :]             # [Hq, 1, D]
        p = torch.softmax(qq @ k.transpose(1, 2) * scale, dim=-1)
        out[b] = (p @ v)[:, 0, :]
    return out.numpy()


def _per_seq(w, fill, deq):
    """Dequantized cache [num_blocks, Hkv, bs, D] -> per-sequence [L, Hkv, D]."""
    bt, bs = fill["block_table"], w.block_size
    res = []
    for b, L in enumerate(w.context_lens):
        p = np.arange(L)
        res.append(deq[bt[b, p // bs], :, p % bs])
    return res


@pytest.mark.parametrize("mode", [orc.BF16, orc.FP8_PER_TENSOR, orc.FP8_PER_HEAD,
                                  orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD])
@pytest.mark.parametrize("window", [0, 16, 50])
def test_decode_matches_torch_attention_on_dequantized_cache(mode, window):
    w = TINY
    fill = host_fill(w)
    sc = np.array([0.05, 0.6], dtype=np.float32) if mode == orc.FP8_PER_HEAD else (
        np.array([1.0], dtype=np.float32) if mode == orc.FP8_PER_TENSOR else None)
    kc, vc, ks, vs = _cache(mode, w, fill, sc)
    q = bits(wl.queries(w, "cpu"))
    got = orc.decode(mode, q, kc, vc, fill["block_table"], fill["context_lens"], k_scale=sc,
                     v_scale=sc, k_cache_scale=ks, v_cache_scale=vs, window=window)
    Kh = _per_seq(w, fill, orc.dequantize(mode, kc, ks, sc))
    Vh = _per_seq(w, fill, orc.dequantize(mode, vc, vs, sc))
    ref = _torch_attention(bf16_to_f64(q), Kh, Vh, fill["context_lens"], w.G, window)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_bf16_layer_equals_float64_attention_on_the_inputs():
    w = TINY
    fill = host_fill(w)
    kc, vc, _, _ = _cache(orc.BF16, w, fill)
    q = bits(wl.queries(w, "cpu"))
    got = orc.decode(orc.BF16, q, kc, vc, fill["block_table"], fill["context_lens"])
    # inputs straight from the generator, sequence-major
    K = bf16_to_f64(fill["k_bits"])
    V = bf16_to_f64(fill["v_bits"])
    starts = np.cumsum([0] + list(w.context_lens))
    Kh = [K[starts[b]:starts[b + 1]] for b in range(w.B)]
    Vh = [V[starts[b]:starts[b + 1]] for b in range(w.B)]
    ref = _torch_attention(bf16_to_f64(q), Kh, Vh, fill["context_lens"], w.G)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_single_position_returns_v0():
    w = TINY
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(orc.FP8_PER_TOKEN_HEAD, w, fill)
    q = bits(wl.queries(w, "cpu"))
    cl = np.array([1, 1], dtype=np.int32)
    got = orc.decode(orc.FP8_PER_TOKEN_HEAD, q, kc, vc, fill["block_table"], cl,
                     k_cache_scale=ks, v_cache_scale=vs)
    Vh = _per_seq(w, fill, orc.dequantize(orc.FP8_PER_TOKEN_HEAD, vc, vs))
    for b in range(2):
        for hq in range(w.Hq):
            assert np.array_equal(got[b, hq], Vh[b][0, hq // w.G])


def test_zero_keys_give_the_mean_of_values():
    w = TINY
    fill = host_fill(w)
    fill["k_bits"] = np.zeros_like(fill["k_bits"])
    kc, vc, ks, vs = _cache(orc.FP8_PER_TOKEN_HEAD, w, fill)
    q = bits(wl.queries(w, "cpu"))
    got = orc.decode(orc.FP8_PER_TOKEN_HEAD, q, kc, vc, fill["block_table"],
                     fill["context_lens"], k_cache_scale=ks, v_cache_scale=vs)
    Vh = _per_seq(w, fill, orc.dequantize(orc.FP8_PER_TOKEN_HEAD, vc, vs))
    for b in range(2):
        mean = Vh[b].mean(axis=0)        # [Hkv, D]
        for hq in range(w.Hq):
            np.testing.assert_allclose(got[b, hq], mean[hq // w.G], rtol=1e-13, atol=1e-13)


def test_window_at_least_context_is_full_attention():
    w = TINY
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(orc.FP8_PER_TOKEN_HEAD, w, fill)
    q = bits(wl.queries(w, "cpu"))
    args = (orc.FP8_PER_TOKEN_HEAD, q, kc, vc, fill["block_table"], fill["context_lens"])
    full = orc.decode(*args, k_cache_scale=ks, v_cache_scale=vs)
    for W in (100, 101, 4096):
        assert np.array_equal(orc.decode(*args, k_cache_scale=ks, v_cache_scale=vs, window=W), full)
    part = orc.decode(*args, k_cache_scale=ks, v_cache_scale=vs, window=99)
    assert np.array_equal(part[0], full[0]) and not np.array_equal(part[1], full[1])


def test_gqa_grouping_uses_kv_head_hq_div_g():
    # V constant per KV head (value h+1) -> every query head of group h returns h+1.
    w = TINY
    fill = host_fill(w)
    v = np.zeros_like(fill["v_bits"])
    for h in range(w.Hkv):
        v[:, h, :] = bits(torch.full((1,), float(h + 1)).to(torch.bfloat16))[0]
    fill["v_bits"] = v
    kc, vc, _, _ = _cache(orc.BF16, w, fill)
    q = bits(wl.queries(w, "cpu"))
    got = orc.decode(orc.BF16, q, kc, vc, fill["block_table"], fill["context_lens"])
    for hq in range(w.Hq):
        np.testing.assert_allclose(got[:, hq], hq // w.G + 1, rtol=0, atol=1e-14)


def test_empty_context_gives_zeros_and_pairs_subset_matches_full():
    w = TINY
    fill = host_fill(w)
    kc, vc, ks, vs = _cache(orc.FP8_PER_TOKEN_HEAD, w, fill)
    q = bits(wl.queries(w, "cpu"))
    cl = np.array([0, 100], dtype=np.int32)
    full = orc.decode(orc.FP8_PER_TOKEN_HEAD, q, kc, vc, fill["block_table"], cl,
                      k_cache_scale=ks, v_cache_scale=vs)
    assert not full[0].any()
    pairs = [(1, 3), (1, 0)]
    sub = orc.decode(orc.FP8_PER_TOKEN_HEAD, q, kc, vc, fill["block_table"], cl,
                     k_cache_scale=ks, v_cache_scale=vs, pairs=pairs)
    assert np.array_equal(sub[0], full[1, 3]) and np.array_equal(sub[1], full[1, 0])


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16])
def test_decode_and_prefill_do_not_depend_on_the_page_size(bs, mode):
    """The same tokens paged in 16-position blocks and in larger ones give the
    same attention: the page size only moves where a position is stored."""
    import dataclasses
    outs = {}
    for size in (16, bs):
        w = dataclasses.replace(TINY, block_size=size)
        fill = host_fill(w)
        kc, vc, ks, vs = orc.alloc_cache(mode, fill["paging"].num_blocks, w.Hkv, size, w.D)
        orc.cache_write(mode, fill["k_bits"], fill["v_bits"], fill["slots_np"], kc, vc, ks, vs,
                        block_size=size)
        q = bits(wl.queries(w, "cpu"))
        dec = orc.decode(mode, q, kc, vc, fill["block_table"], fill["context_lens"],
                         k_cache_scale=ks, v_cache_scale=vs, window=20, block_size=size)
        qs = np.array([0, 10, 60], dtype=np.int32)
        qp = bits(wl.kv_tokens(w, 60, "cpu", stream_base=703)[0][:, :1].expand(-1, w.Hq, -1)
                  .contiguous())
        pre = orc.prefill(mode, qp, kc, vc, fill["block_table"], qs, fill["context_lens"],
                          k_cache_scale=ks, v_cache_scale=vs, block_size=size)
        outs[size] = (dec, pre)
    assert np.array_equal(outs[16][0], outs[bs][0])
    assert np.array_equal(outs[16][1], outs[bs][1])
