"""Python face of the CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It wraps ``kvq_oracle.c`` (compiled here
with gcc into ``liborcl.so``) with numpy arrays, and shares nothing with the
CUDA library: it has its own copy of the mode numbers and of the cache-layout
arithmetic, written from the same layout contract.

Parity pinned: the codec (exhaustive and against the printed E4M3 format and
torch's float8 cast), the write (amax invariant, zero-vector rule, skipped
slots, plain-cast special case, closed-form error bound, hand-worked bytes
of INT4 packing and FP8 codes), the decode
(library softmax attention for BF16 layers, L = 1, K = 0, window >= L), the
prefill (masked library attention, causal and window) and the FP8 query
(torch's E4M3 cast, ties and saturation) are all checked against facts that
do not come from this module; see tests/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvq_oracle.c")
LIB = os.path.join(HERE, "liborcl.so")

# Mode numbers of the oracle (same values as the library's public enum, by
# contract: 0 BF16, 1 FP8 per-tensor, 2 FP8 static per-head, 3 FP8 dynamic
# per-token-head, 4 packed INT4 per-token-head).
BF16, FP8_PER_TENSOR, FP8_PER_HEAD, FP8_PER_TOKEN_HEAD, INT4_PER_TOKEN_HEAD = range(5)
DYNAMIC_MODES = (FP8_PER_TOKEN_HEAD, INT4_PER_TOKEN_HEAD)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c with gcc (OpenMP, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            P = ctypes.c_void_p
            i32, i64, f32, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_double
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [f32]
            L.orc_e4m3_encode_array.restype = None
            L.orc_e4m3_encode_array.argtypes = [P, P, i64]
            L.orc_e4m3_decode.restype = f64
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_int4_encode.restype = i32
            L.orc_int4_encode.argtypes = [f32]
            L.orc_cache_write.restype = i32
            L.orc_cache_write.argtypes = [i32, i64, i32, i32, i32, i64, P, P, P, P, P, P, P, P, P]
            L.orc_calibrate_per_head.restype = None
            L.orc_calibrate_per_head.argtypes = [i64, i32, i32, P, f32, P]
            L.orc_decode_pairs.restype = i32
            L.orc_decode_pairs.argtypes = [i32, i32, i32, i32, i32, i64, i32, f64, P, P, P, P, P,
                                           P, P, P, i32, P, i32, P, P, P]
            L.orc_num_threads.restype = i32
            L.orc_set_num_threads.argtypes = [i32]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- codec
def e4m3_encode(y: float) -> int:
    return int(lib().orc_e4m3_encode(float(y)))


def e4m3_decode(c: int) -> float:
    return float(lib().orc_e4m3_decode(int(c)))


def int4_encode(y: float) -> int:
    return int(lib().orc_int4_encode(float(y)))


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


# ---------------------------------------------------------------- layout
def row_bytes(mode: int, D: int) -> int:
    if mode == BF16:
        return 2 * D
    if mode == INT4_PER_TOKEN_HEAD:
        return D // 2
    return D


def alloc_cache(mode: int, num_blocks: int, Hkv: int, bs: int, D: int):
    """Zeroed host cache for one layer: (k_codes, v_codes, k_scales, v_scales)."""
    rb = row_bytes(mode, D)
    kc = np.zeros((num_blocks, Hkv, bs, rb), dtype=np.uint8)
    vc = np.zeros_like(kc)
    if mode in DYNAMIC_MODES:
        ks = np.zeros((num_blocks, Hkv, bs), dtype=np.float32)
        vs = np.zeros_like(ks)
    else:
        ks = vs = None
    return kc, vc, ks, vs


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 arrays are passed as their uint16 bit patterns"
    return a


# ---------------------------------------------------------------- write
def cache_write(mode, k_new, v_new, slot_mapping, k_cache, v_cache, k_cache_scale=None,
                v_cache_scale=None, k_scale=None, v_scale=None, block_size=16):
    """Quantize bf16 K/V [T, Hkv, D] (uint16 bits) into the host cache in place."""
    k_new, v_new = _u16(k_new), _u16(v_new)
    T, Hkv, D = k_new.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    num_blocks = k_cache.shape[0]
    rc = lib().orc_cache_write(mode, T, Hkv, D, block_size, num_blocks, _ptr(k_new), _ptr(v_new),
                               _ptr(slots), _ptr(ks), _ptr(vs), _ptr(k_cache), _ptr(v_cache),
                               _ptr(k_cache_scale), _ptr(v_cache_scale))
    if rc != 0:
        raise ValueError("oracle cache_write: slot outside the cache")


def calibrate_per_head(x, qmax=448.0):
    x = _u16(x)
    T, Hkv, D = x.shape
    out = np.zeros(Hkv, dtype=np.float32)
    lib().orc_calibrate_per_head(T, Hkv, D, _ptr(x), float(qmax), _ptr(out))
    return out


# ---------------------------------------------------------------- decode
def decode(mode, q, k_cache, v_cache, block_table, context_lens, *, k_scale=None, v_scale=None,
           k_cache_scale=None, v_cache_scale=None, window=0, softmax_scale=0.0, block_size=16,
           pairs=None):
    """float64 decode attention.  q is [B, Hq, D] uint16 (bf16 bits).

    Returns [B, Hq, D] float64, or [len(pairs), D] when ``pairs`` (a list of
    (b, hq)) is given.
    """
    q = _u16(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    if softmax_scale == 0.0:
        softmax_scale = 1.0 / np.sqrt(D)
    if pairs is None:
        pb = np.repeat(np.arange(B, dtype=np.int32), Hq)
        ph = np.tile(np.arange(Hq, dtype=np.int32), B)
    else:
        pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
        pb, ph = np.ascontiguousarray(pairs[:, 0]), np.ascontiguousarray(pairs[:, 1])
    out = np.zeros((len(pb), D), dtype=np.float64)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    rc = lib().orc_decode_pairs(mode, Hq, Hkv, D, block_size, k_cache.shape[0], int(window),
                                float(softmax_scale), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                _ptr(ks), _ptr(vs), _ptr(k_cache_scale), _ptr(v_cache_scale),
                                _ptr(bt), bt.shape[1], _ptr(cl), len(pb), _ptr(pb), _ptr(ph),
                                _ptr(out))
    if rc != 0:
        raise ValueError("oracle decode: block-table entry outside the cache")
    return out.reshape(B, Hq, D) if pairs is None else out


def prefill(mode, q, k_cache, v_cache, block_table, query_start, context_lens, *, pairs=None,
            **kw):
    """float64 prefill attention: row query_start[b] + i of q (bf16 bits
    [T, Hq, D]) is the query at position p = L_b - n_b + i of sequence b, and
    its output is the decode of that query with context p + 1 (positions
    [lo(p), p], causal; the window and scales as in decode).  Returns
    [T, Hq, D], or [len(pairs), D] for pairs (token, hq)."""
    q = _u16(q)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    qs = np.asarray(query_start, dtype=np.int64)
    cl = np.asarray(context_lens, dtype=np.int64)
    T = int(qs[-1])
    seq = np.zeros(T, dtype=np.int64)
    ctx = np.zeros(T, dtype=np.int32)
    for b in range(len(cl)):
        n = int(qs[b + 1] - qs[b])
        if n <= 0:
            continue
        seq[qs[b]:qs[b + 1]] = b
        ctx[qs[b]:qs[b + 1]] = int(cl[b]) - n + 1 + np.arange(n)
    return decode(mode, q, k_cache, v_cache, bt[seq], ctx, pairs=pairs, **kw)


def quantize_query(q, q_scale):
    """FP8 query of the Q-scale path (the pages' per-tensor FP8 with one Q
    scale, or one Q scale per query head: [P3] "FP8 KV cache layer skipping vs
    per-head scales", opening section).  Each element x of q (bf16 bits
    [B, Hq, D]) becomes the E4M3 code of y = RN32(x / s) (IEEE fp32 division,
    then round to nearest even, saturating), s = q_scale[0] or q_scale[hq].
    Returns the bf16 bits of the codes' values (E4M3 values are exact in
    bf16) and the per-head scales [Hq] as float64."""
    q = _u16(q)
    B, Hq, D = q.shape
    qs = np.asarray(q_scale, dtype=np.float32).reshape(-1)
    s = np.broadcast_to(qs, (Hq,)) if qs.size == 1 else qs
    x = (q.astype(np.uint32) << 16).view(np.float32)
    y = np.ascontiguousarray(x / s[None, :, None], dtype=np.float32)   # fp32 RN division
    codes = np.empty(y.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(y.ctypes.data, codes.ctypes.data, y.size)
    vals = e4m3_decode_table()[codes].astype(np.float32)
    return (vals.view(np.uint32) >> 16).astype(np.uint16), s.astype(np.float64)


def decode_fp8_query(mode, q, q_scale, k_cache, v_cache, block_table, context_lens, *,
                     softmax_scale=0.0, pairs=None, **kw):
    """float64 decode with the FP8 query q_hat = E4M3(q / s) x s: the scores
    are softmax_scale x s x <E4M3 value, K_hat>, so each query head is decoded
    with its own factor.  Same returns as decode."""
    codes, s = quantize_query(q, q_scale)
    B, Hq, D = codes.shape
    if softmax_scale == 0.0:
        softmax_scale = 1.0 / np.sqrt(D)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(Hq)]
    pairs = [tuple(p) for p in pairs]
    out = np.zeros((len(pairs), D), dtype=np.float64)
    for h in sorted(set(p[1] for p in pairs)):
        idx = [i for i, p in enumerate(pairs) if p[1] == h]
        out[idx] = decode(mode, codes, k_cache, v_cache, block_table, context_lens,
                          softmax_scale=float(softmax_scale * s[h]),
                          pairs=[pairs[i] for i in idx], **kw)
    return out


def dequantize(mode, k_cache, k_cache_scale=None, k_scale=None):
    """Dequantized cache values [num_blocks, Hkv, bs, D] in float64 (for tests)."""
    table = e4m3_decode_table()
    if mode == BF16:
        u = k_cache.view(np.uint16).astype(np.uint32) << 16
        return u.view(np.float32).astype(np.float64)
    if mode == INT4_PER_TOKEN_HEAD:
        lo = (k_cache & 0xF).astype(np.int64)
        hi = (k_cache >> 4).astype(np.int64)
        lo = np.where(lo >= 8, lo - 16, lo)
        hi = np.where(hi >= 8, hi - 16, hi)
        vals = np.stack([lo, hi], axis=-1).reshape(*k_cache.shape[:-1], -1).astype(np.float64)
        return vals * k_cache_scale[..., None].astype(np.float64)
    vals = table[k_cache]
    if mode == FP8_PER_TENSOR:
        return vals * float(k_scale[0])
    if mode == FP8_PER_HEAD:
        return vals * np.asarray(k_scale, dtype=np.float64)[None, :, None, None]
    return vals * k_cache_scale[..., None].astype(np.float64)
