"""The decode tolerance must reject the precision mistakes a kernel could make.

tests/helpers.check_attention (with attention_tolerance) is the bar every
GPU decode case is held to.  These CPU tests show, on the Llama-8B-like
recipe (per-KV-head multipliers log-uniform in [0.5, 32], 1% of positions
x8, dynamic per-token-head FP8, full 4096-position contexts), that the bar
is discriminating: a float64 decode on the dequantized cache that makes one
plausible shortcut fails it, while the same decode with the split the
kernels use passes.

Shortcuts simulated, each otherwise exact (float64):
  * the weight that meets V, P' = p * v_scale * 2^k, rounded to one f16
    (11 significant bits) instead of the f16 hi + lo pair (about 22 bits);
  * K dequantized to bf16 (code x scale rounded to 8 significant bits)
    before the dot product;
  * the score rounded to f16 before the exponent.
The two-term split and a score rounded to fp32 must pass.
"""
import numpy as np
import pytest

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.helpers import attention_tolerance, bf16_to_f64, bits, check_attention, host_fill

W = wl.scaled(wl.CONFIGS["llama8b"], batch=2, context=4096)
KP = 13          # P' < 2^14 (the kernels' range factor)


@pytest.fixture(scope="module")
def case():
    w = W
    fill = host_fill(w)
    mode = orc.FP8_PER_TOKEN_HEAD
    pg = fill["paging"]
    kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, w.Hkv, w.block_size, w.D)
    orc.cache_write(mode, fill["k_bits"], fill["v_bits"], fill["slots_np"], kc, vc, ks, vs)
    q = bits(wl.queries(w, "cpu"))
    ref = orc.decode(mode, q, kc, vc, fill["block_table"], fill["context_lens"],
                     k_cache_scale=ks, v_cache_scale=vs)
    table = orc.e4m3_decode_table()
    bt, bs = fill["block_table"], w.block_size
    rows = []
    for b in range(w.B):
        L = int(fill["context_lens"][b])
        p = np.arange(L)
        blk, off = bt[b, p // bs], p % bs
        for g in range(w.Hkv):
            kcode = table[kc[blk, g, off]]                       # [L, D] code values
            vcode = table[vc[blk, g, off]]
            ksc = ks[blk, g, off].astype(np.float64)
            vsc = vs[blk, g, off].astype(np.float64)
            rows.append((b, g, kcode, vcode, ksc, vsc))
    return dict(w=w, q=bf16_to_f64(q), ref=ref, rows=rows)


def _decode(case, score_round=None, k_round=None, weight_split=None):
    """float64 decode with one step rounded as the simulated kernel would."""
    w, qd = case["w"], case["q"]
    scale = 1.0 / np.sqrt(w.D)
    out = np.zeros_like(case["ref"])
    tol = np.zeros_like(case["ref"])
    for b, g, kcode, vcode, ksc, vsc in case["rows"]:
        Kh = kcode * ksc[:, None]
        Vh = vcode * vsc[:, None]
        Kq = k_round(Kh) if k_round else Kh
        vexp = int(np.floor(np.log2(vsc.max())))
        for j in range(w.G):
            hq = g * w.G + j
            s = (Kq @ qd[b, hq]) * scale
            if score_round:
                s = score_round(s)
            pr = np.exp(s - s.max())
            pp = pr * vsc * 2.0 ** (KP - vexp)                  # P' < 2^14
            if weight_split:
                pp = weight_split(pp)
            out[b, hq] = (pp @ vcode) / pr.sum() * 2.0 ** (vexp - KP)
            tol[b, hq] = attention_tolerance(qd[b, hq], Kh, Vh, case["ref"][b, hq], scale)
    return out, tol


def _f16(x):
    return x.astype(np.float16).astype(np.float64)


def _f16_hi_lo(x):
    hi = _f16(x)
    return hi + _f16(x - hi)


def _bf16(x):
    # round to nearest even on the float32 bit pattern, keep the top 16 bits
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _fp32(x):
    return x.astype(np.float32).astype(np.float64)


def test_split_weight_and_fp32_scores_pass(case):
    out, tol = _decode(case, score_round=_fp32, weight_split=_f16_hi_lo)
    check_attention(out, case["ref"], tol, "two-term P' split, fp32 scores")


def test_single_f16_weight_is_rejected(case):
    out, tol = _decode(case, weight_split=_f16)
    with pytest.raises(AssertionError, match="over tolerance"):
        check_attention(out, case["ref"], tol, "P' as one f16")


def test_bf16_dequantized_keys_are_rejected(case):
    out, tol = _decode(case, k_round=_bf16, weight_split=_f16_hi_lo)
    with pytest.raises(AssertionError, match="over tolerance"):
        check_attention(out, case["ref"], tol, "K rounded to bf16")


def test_f16_scores_are_rejected(case):
    out, tol = _decode(case, score_round=_f16, weight_split=_f16_hi_lo)
    with pytest.raises(AssertionError, match="over tolerance|relative L2"):
        check_attention(out, case["ref"], tol, "scores rounded to f16")


def test_flat_bound_is_beyond_fp32_scores_on_the_full_llama8b_recipe():
    """Why the Llama-8B-like rows are held to the per-row bound and not the
    flat 2e-3: on the full workload (64 sequences x 4096 positions), a decode
    whose only rounding is each score rounded once to fp32 (everything else
    float64) already misses 2e-3 on some rows, where near-tied scores of
    several hundred select values of several hundred.  No kernel with fp32
    scores can do better.  The per-row bound accepts it."""
    w = wl.CONFIGS["llama8b"]
    fill = host_fill(w)
    mode = orc.FP8_PER_TOKEN_HEAD
    pg = fill["paging"]
    kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, w.Hkv, w.block_size, w.D)
    orc.cache_write(mode, fill["k_bits"], fill["v_bits"], fill["slots_np"], kc, vc, ks, vs)
    qd = bf16_to_f64(bits(wl.queries(w, "cpu")))
    Kh = orc.dequantize(mode, kc, ks)
    Vh = orc.dequantize(mode, vc, vs)
    bt, bs = fill["block_table"], w.block_size
    scale = 1.0 / np.sqrt(w.D)
    worst, rows_over = 0.0, 0
    for b in range(w.B):
        p = np.arange(int(fill["context_lens"][b]))
        blk, off = bt[b, p // bs], p % bs
        for g in range(w.Hkv):
            K, V = Kh[blk, g, off], Vh[blk, g, off]
            for j in range(w.G):
                q = qd[b, g * w.G + j]
                s = (K @ q) * scale
                e = np.exp(s - s.max())
                ref = (e @ V) / e.sum()
                s32 = s.astype(np.float32).astype(np.float64)
                e32 = np.exp(s32 - s32.max())
                got = (e32 @ V) / e32.sum()
                err = np.abs(got - ref)
                if err.max() > 2e-3:
                    rows_over += 1
                    assert np.all(err <= attention_tolerance(q, K, V, ref, scale))
                worst = max(worst, float(err.max()))
    assert rows_over > 0 and worst > 2e-3
