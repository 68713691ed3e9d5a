"""Capacity and metadata accounting, written out from the pages' formulas.

Test infrastructure only (see oracle.py).  Each function restates one formula;
the tests pin them to the worked numbers the pages print.
"""
from __future__ import annotations


def payload_bytes_per_token(layers: int, kv_heads: int, head_size: float, bytes_per_elem: float):
    """2 x layers x KV heads x head size x bytes per element.

    "Per-token-head KV cache scale overhead", section "Per-token-head KV cache
    scale overhead" (the ordinary KV cache formula; the 2 is K and V).
    """
    return 2 * layers * kv_heads * head_size * bytes_per_elem


def dynamic_scale_bytes_per_token(layers: int, kv_heads: int, scale_bytes: int = 4):
    """2 x layers x KV heads x 4 bytes: one FP32 K and one FP32 V scale per
    layer and KV head at every token position; no head-size term.

    "Per-token-head KV cache scale overhead", section "Per-token-head KV cache
    scale overhead".
    """
    return 2 * layers * kv_heads * scale_bytes


def fp8_scale_tax(head_size: int) -> float:
    """8 / (2 x head size) = 4 / head size.

    "Per-token-head KV cache scale overhead", section "The FP8 scale tax is 4
    divided by head size".
    """
    return 8.0 / (2.0 * head_size)


def int4_scale_tax(head_size: int) -> float:
    """8 / head size: packed INT4 K and V use one head size of bytes per
    layer and KV head, and the two FP32 scales still add 8 bytes.

    "Per-token-head KV cache scale overhead", section "INT4 makes the metadata
    fraction larger".
    """
    return 8.0 / head_size


def per_tensor_metadata_bytes(layers: int, scale_bytes: int = 4) -> int:
    """K and V only: layers x 2 x 4 bytes.

    "Per-tensor vs per-head FP8 KV cache scales", section "Static per-head
    metadata is almost free".
    """
    return layers * 2 * scale_bytes


def static_per_head_metadata_bytes(layers: int, kv_heads: int, scale_bytes: int = 4) -> int:
    """K and V only: layers x KV heads x 2 x 4 bytes (same section)."""
    return layers * kv_heads * 2 * scale_bytes


def static_per_head_extra_bytes_with_q(q_heads: int, kv_heads: int, scale_bytes: int = 4) -> int:
    """Per layer, per-head shapes hold H + 2 Hkv scales against 3 per-tensor
    scales (Q, K, V): extra = 4 (H + 2 Hkv - 3) bytes.

    "FP8 KV cache layer skipping vs per-head scales", section "Per-head scales
    have fixed overhead".
    """
    return scale_bytes * (q_heads + 2 * kv_heads - 3)


def static_per_head_scale_count_with_q(q_heads: int, kv_heads: int) -> int:
    return q_heads + 2 * kv_heads


def retained_positions(context: int, window: int) -> int:
    """A full layer retains the context; a sliding layer retains at most W.

    "FP8 KV cache layer skipping vs per-head scales", section "Layer skipping
    follows retained-token footprint".
    """
    return context if window <= 0 else min(context, window)


def skip_accounting(context: int, windows, skipped, kv_heads: int, head_size: int):
    """All-FP8 bytes C*A, mixed FP8/BF16 bytes C*(A+S), compression 2A/(A+S).

    C = 2 x KV heads x head size at one byte per element; A = retained
    positions over every layer, S = over the skipped layers only.  Same page,
    section "Layer skipping follows retained-token footprint".
    """
    A = sum(retained_positions(context, w) for w in windows)
    S = sum(retained_positions(context, w) for w, s in zip(windows, skipped) if s)
    C = 2 * kv_heads * head_size
    return {
        "A": A,
        "S": S,
        "C": C,
        "bf16_bytes": 2 * C * A,
        "fp8_bytes": C * A,
        "mixed_bytes": C * (A + S),
        "compression": 2 * A / (A + S),
    }


def block_bytes(bytes_per_token: float, block_size: int) -> float:
    """Bytes per token x block size, before allocator alignment.

    "Per-token-head KV cache scale overhead", section "Convert bytes into
    block capacity".
    """
    return bytes_per_token * block_size
