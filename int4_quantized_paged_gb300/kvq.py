"""Thin ctypes binding of libkvq (include/kvq.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  Tensors are
passed as raw device pointers (``tensor.data_ptr()``); torch provides device
memory and streams, nothing else.  Importing this module loads libkvq.so and
raises ImportError when it has not been built -- there is no other path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libkvq.so is not built ({LIB_PATH}); run "
                      "`python -m int4_quantized_paged_gb300.build` or __graft_entry__.build()")
_lib = ctypes.CDLL(LIB_PATH)

BF16, FP8_PER_TENSOR, FP8_PER_HEAD, FP8_PER_TOKEN_HEAD, INT4_PER_TOKEN_HEAD = range(5)
MODE_NAMES = {"bf16": BF16, "fp8_per_tensor": FP8_PER_TENSOR, "fp8_per_head": FP8_PER_HEAD,
              "fp8_per_token_head": FP8_PER_TOKEN_HEAD, "int4_per_token_head": INT4_PER_TOKEN_HEAD}
DYNAMIC = (FP8_PER_TOKEN_HEAD, INT4_PER_TOKEN_HEAD)
STATUS = ["KVQ_OK", "KVQ_ERR_INVALID_ARG", "KVQ_ERR_UNSUPPORTED", "KVQ_ERR_ALIGNMENT",
          "KVQ_ERR_WORKSPACE", "KVQ_ERR_CUDA", "KVQ_ERR_BAD_INDEX", "KVQ_ERR_TIMEOUT"]

P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_size_t


class kvq_config(ctypes.Structure):
    _fields_ = [("num_layers", i32), ("num_q_heads", i32), ("num_kv_heads", i32),
                ("head_dim", i32), ("block_size", i32), ("num_blocks", i64),
                ("layer_mode", ctypes.POINTER(i32)), ("layer_window", ctypes.POINTER(i32)),
                ("softmax_scale", f32)]


class kvq_capacity(ctypes.Structure):
    _fields_ = [("payload_bytes_per_token", ctypes.c_double),
                ("scale_bytes_per_token", ctypes.c_double),
                ("bytes_per_token", ctypes.c_double), ("block_bytes", ctypes.c_double),
                ("retained_positions", i64), ("static_scale_bytes", i64),
                ("cache_bytes", ctypes.c_double), ("bf16_cache_bytes", ctypes.c_double)]


_SIGS = {
    "kvq_create": (i32, [ctypes.POINTER(kvq_config), ctypes.POINTER(P)]),
    "kvq_destroy": (None, [P]),
    "kvq_layer_buffer_sizes": (i32, [P, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
    "kvq_cache_bytes": (i32, [P, i64, ctypes.POINTER(kvq_capacity)]),
    "kvq_cache_write": (i32, [P, i32, P, P, i64, P, i64, P, P, P, P, P, P, P]),
    "kvq_calibrate_per_head": (i32, [P, P, i64, f32, P, P]),
    "kvq_decode_plan": (i32, [P, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(sz)]),
    "kvq_decode_workspace_size": (sz, [P, i32, i32, i32]),
    "kvq_decode_attention": (i32, [P, i32, P, P, P, P, P, P, P, P, i32, P, i32, i32, P, i32, P,
                                   sz, P]),
    "kvq_prefill_attention": (i32, [P, i32, P, P, P, P, P, P, P, P, i32, P, P, i32, i32, P, P]),
    "kvq_decode_attention_fp8_query": (i32, [P, i32, P, P, i32, P, P, P, P, P, P, P, i32, P, i32,
                                             i32, P, i32, P, sz, P]),
    "kvq_decode_attention_bf16": (i32, [P, i32, P, P, P, P, P, P, P, P, i32, P, i32, i32, P, i32,
                                        P, sz, P]),
    "kvq_decode_attention_fixed_scratch": (i32, [P, i32, P, P, P, P, P, P, P, P, i32, P, i32,
                                                 i32, P, i32, P]),
    "kvq_e4m3_encode": (i32, [P, P, i64, P]),
    "kvq_get_device_error": (i32, [P]),
    "kvq_check_bounded_wait": (i32, [i64, P]),
    "kvq_status_string": (ctypes.c_char_p, [i32]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS[status] if 0 <= status < len(STATUS) else str(status)
        msg = _lib.kvq_status_string(status).decode()
        super().__init__(f"{where}: {name} ({msg})")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise KVQError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Context:
    """Owns a kvq_ctx handle (host-only configuration)."""

    def __init__(self, handle: int, cfg: dict):
        self.handle = handle
        self.cfg = cfg

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            _lib.kvq_destroy(h)

    @property
    def _as_parameter_(self):
        return ctypes.c_void_p(self.handle)


def kvq_create(num_layers: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
               block_size: int, num_blocks: int, layer_mode: Sequence[int],
               layer_window: Optional[Sequence[int]] = None, softmax_scale: float = 0.0) -> Context:
    modes = (i32 * num_layers)(*[int(m) for m in layer_mode])
    wins = None if layer_window is None else (i32 * num_layers)(*[int(w) for w in layer_window])
    cfg = kvq_config(num_layers, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     ctypes.cast(modes, ctypes.POINTER(i32)),
                     None if wins is None else ctypes.cast(wins, ctypes.POINTER(i32)),
                     softmax_scale)
    h = P()
    _check(_lib.kvq_create(ctypes.byref(cfg), ctypes.byref(h)), "kvq_create")
    return Context(h.value, dict(num_layers=num_layers, Hq=num_q_heads, Hkv=num_kv_heads,
                                 D=head_dim, block_size=block_size, num_blocks=num_blocks,
                                 layer_mode=list(layer_mode),
                                 layer_window=list(layer_window or [0] * num_layers)))


def kvq_layer_buffer_sizes(ctx: Context, layer: int):
    c, s = sz(), sz()
    _check(_lib.kvq_layer_buffer_sizes(ctx, layer, ctypes.byref(c), ctypes.byref(s)),
           "kvq_layer_buffer_sizes")
    return c.value, s.value


def kvq_cache_bytes(ctx: Context, context_tokens: int) -> dict:
    r = kvq_capacity()
    _check(_lib.kvq_cache_bytes(ctx, context_tokens, ctypes.byref(r)), "kvq_cache_bytes")
    return {f: getattr(r, f) for f, _ in kvq_capacity._fields_}


def alloc_layer_cache(ctx: Context, layer: int, device="cuda"):
    """Device buffers for one layer: (k_codes, v_codes, k_scales, v_scales); the
    scale tensors are None for non-dynamic modes.  Shapes follow the layout."""
    c = ctx.cfg
    code_b, scale_b = kvq_layer_buffer_sizes(ctx, layer)
    rows = c["num_blocks"] * c["Hkv"] * c["block_size"]
    rb = code_b // max(rows, 1) if rows else 0
    shape = (c["num_blocks"], c["Hkv"], c["block_size"], rb)
    kc = torch.zeros(shape, dtype=torch.uint8, device=device)
    vc = torch.zeros(shape, dtype=torch.uint8, device=device)
    if scale_b:
        ks = torch.zeros(shape[:3], dtype=torch.float32, device=device)
        vs = torch.zeros(shape[:3], dtype=torch.float32, device=device)
    else:
        ks = vs = None
    return kc, vc, ks, vs


def kvq_cache_write(ctx: Context, layer: int, k_new, v_new, slot_mapping, k_cache, v_cache,
                    k_cache_scale=None, v_cache_scale=None, k_scale=None, v_scale=None,
                    kv_token_stride: int = 0, num_tokens: Optional[int] = None, stream=None):
    T = k_new.shape[0] if num_tokens is None else num_tokens
    _check(_lib.kvq_cache_write(ctx, layer, _ptr(k_new), _ptr(v_new), kv_token_stride,
                                _ptr(slot_mapping), T, _ptr(k_scale), _ptr(v_scale),
                                _ptr(k_cache), _ptr(v_cache), _ptr(k_cache_scale),
                                _ptr(v_cache_scale), _stream(stream)), "kvq_cache_write")


def kvq_calibrate_per_head(ctx: Context, x, scale_out, qmax: float = 448.0,
                           num_tokens: Optional[int] = None, stream=None):
    T = x.shape[0] if num_tokens is None else num_tokens
    _check(_lib.kvq_calibrate_per_head(ctx, _ptr(x), T, qmax, _ptr(scale_out), _stream(stream)),
           "kvq_calibrate_per_head")


def kvq_decode_plan(ctx: Context, layer: int, batch: int, max_context: int, num_workers: int = 0):
    s, w = i32(num_workers), sz()
    _check(_lib.kvq_decode_plan(ctx, layer, batch, max_context, ctypes.byref(s), ctypes.byref(w)),
           "kvq_decode_plan")
    return s.value, w.value


def kvq_decode_workspace_size(ctx: Context, layer: int, batch: int, max_context: int) -> int:
    return int(_lib.kvq_decode_workspace_size(ctx, layer, batch, max_context))


def kvq_decode_attention(ctx: Context, layer: int, q, k_cache, v_cache, block_table,
                         context_lens, out, *, max_context: int, k_scale=None, v_scale=None,
                         k_cache_scale=None, v_cache_scale=None, num_workers: int = 0,
                         workspace=None, workspace_bytes: Optional[int] = None,
                         batch: Optional[int] = None, max_blocks_per_seq: Optional[int] = None,
                         stream=None):
    B = q.shape[0] if batch is None else batch
    mb = block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.kvq_decode_attention(ctx, layer, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(k_cache_scale),
                                     _ptr(v_cache_scale), _ptr(block_table), mb,
                                     _ptr(context_lens), B, max_context, _ptr(out), num_workers,
                                     _ptr(workspace), workspace_bytes, _stream(stream)),
           "kvq_decode_attention")


def kvq_prefill_attention(ctx: Context, layer: int, q, k_cache, v_cache, block_table,
                          query_start, context_lens, out, *, max_query_len: int, k_scale=None,
                          v_scale=None, k_cache_scale=None, v_cache_scale=None,
                          batch: Optional[int] = None, max_blocks_per_seq: Optional[int] = None,
                          stream=None):
    """Causal attention of each sequence's new tokens (rows of q between
    query_start[b] and query_start[b+1]) over the cache; see include/kvq.h."""
    B = context_lens.shape[0] if batch is None else batch
    mb = block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq
    _check(_lib.kvq_prefill_attention(ctx, layer, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(k_cache_scale),
                                      _ptr(v_cache_scale), _ptr(block_table), mb,
                                      _ptr(query_start), _ptr(context_lens), B, max_query_len,
                                      _ptr(out), _stream(stream)), "kvq_prefill_attention")


def kvq_decode_attention_fp8_query(ctx: Context, layer: int, q, q_scale, k_cache, v_cache,
                                   block_table, context_lens, out, *, max_context: int,
                                   k_scale=None, v_scale=None, k_cache_scale=None,
                                   v_cache_scale=None, num_workers: int = 0, workspace=None,
                                   workspace_bytes: Optional[int] = None,
                                   batch: Optional[int] = None,
                                   max_blocks_per_seq: Optional[int] = None, stream=None):
    """kvq_decode_attention with the query quantized to E4M3 by q_scale (a
    device fp32 tensor of 1 or Hq scales)."""
    B = q.shape[0] if batch is None else batch
    mb = block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.kvq_decode_attention_fp8_query(
        ctx, layer, _ptr(q), _ptr(q_scale), 0 if q_scale is None else q_scale.numel(),
        _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale), _ptr(v_scale), _ptr(k_cache_scale), _ptr(v_cache_scale),
        _ptr(block_table), mb, _ptr(context_lens), B, max_context, _ptr(out), num_workers,
        _ptr(workspace), workspace_bytes, _stream(stream)), "kvq_decode_attention_fp8_query")


def kvq_decode_attention_bf16(ctx: Context, layer: int, q, k_cache, v_cache, block_table,
                              context_lens, out, *, max_context: int, k_scale=None, v_scale=None,
                              k_cache_scale=None, v_cache_scale=None, num_workers: int = 0,
                              workspace=None, workspace_bytes: Optional[int] = None,
                              batch: Optional[int] = None,
                              max_blocks_per_seq: Optional[int] = None, stream=None):
    """kvq_decode_attention writing a bf16 [B, Hq, D] output."""
    B = q.shape[0] if batch is None else batch
    mb = block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.kvq_decode_attention_bf16(ctx, layer, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_scale), _ptr(v_scale), _ptr(k_cache_scale),
                                          _ptr(v_cache_scale), _ptr(block_table), mb,
                                          _ptr(context_lens), B, max_context, _ptr(out),
                                          num_workers, _ptr(workspace), workspace_bytes,
                                          _stream(stream)),
           "kvq_decode_attention_bf16")


def kvq_decode_attention_fixed_scratch(ctx: Context, layer: int, q, k_cache, v_cache,
                                       block_table, context_lens, out, *, max_context: int,
                                       k_scale=None, v_scale=None, k_cache_scale=None,
                                       v_cache_scale=None, num_workers: int = 0,
                                       batch: Optional[int] = None,
                                       max_blocks_per_seq: Optional[int] = None, stream=None):
    """Decode attention with the library's static scratch instead of a caller
    workspace (see include/kvq.h); nothing is allocated."""
    B = q.shape[0] if batch is None else batch
    mb = block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq
    _check(_lib.kvq_decode_attention_fixed_scratch(
        ctx, layer, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(k_cache_scale), _ptr(v_cache_scale), _ptr(block_table), mb, _ptr(context_lens), B,
        max_context, _ptr(out), num_workers, _stream(stream)), "kvq_decode_attention_fixed_scratch")


def kvq_e4m3_encode(x, out, n: Optional[int] = None, stream=None):
    _check(_lib.kvq_e4m3_encode(_ptr(x), _ptr(out), x.numel() if n is None else n,
                                _stream(stream)), "kvq_e4m3_encode")


def kvq_get_device_error(stream=None) -> int:
    """Synchronizes the stream; returns (and clears) the device error status."""
    return int(_lib.kvq_get_device_error(_stream(stream)))


def kvq_check_bounded_wait(limit_cycles: int, stream=None):
    """Enqueues one warp whose bounded barrier wait runs out after
    limit_cycles SM cycles and sets the TIMEOUT bit (see include/kvq.h)."""
    _check(_lib.kvq_check_bounded_wait(int(limit_cycles), _stream(stream)),
           "kvq_check_bounded_wait")


def kvq_status_string(status: int) -> str:
    return _lib.kvq_status_string(status).decode()
