"""Pins for the capacity/metadata formulas: the worked numbers on the pages
(tests/golden/accounting.json, each entry citing its page and section)."""
import json
import os

import pytest

from oracle import accounting as acc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "accounting.json")))
GiB, MiB, KiB = 2 ** 30, 2 ** 20, 2 ** 10


def test_80_layer_128k_example():
    g = GOLD["fp8_80_layer_128k"]
    L, H, D, T = g["layers"], g["kv_heads"], g["head_size"], g["context"]
    assert acc.per_tensor_metadata_bytes(L) == g["per_tensor_metadata_bytes"]
    assert acc.static_per_head_metadata_bytes(L, H) == g["static_per_head_metadata_bytes"]
    assert (acc.static_per_head_metadata_bytes(L, H) - acc.per_tensor_metadata_bytes(L)
            == g["metadata_difference_bytes"])
    fp8 = acc.payload_bytes_per_token(L, H, D, 1) * T
    assert fp8 == g["fp8_kv_bytes"] and fp8 / GiB == g["fp8_kv_gib"]
    sc = acc.dynamic_scale_bytes_per_token(L, H) * T
    assert sc == g["dynamic_scale_bytes"] and sc / MiB == g["dynamic_scale_mib"]
    assert (fp8 + sc) / GiB == g["fp8_plus_scales_gib"]
    assert acc.payload_bytes_per_token(L, H, D, 2) * T / GiB == g["bf16_kv_gib"]
    assert 2 * D == g["fp8_data_bytes_per_token_head_pair"]
    assert acc.dynamic_scale_bytes_per_token(1, 1) == g["scale_bytes_per_token_head_pair"]
    assert acc.fp8_scale_tax(D) == g["scale_fraction"]


def test_32_layer_gqa_example():
    g = GOLD["gqa_32_layer"]
    L, H, D, T, bs = g["layers"], g["kv_heads"], g["head_size"], g["context"], g["block_size"]
    pay = acc.payload_bytes_per_token(L, H, D, 1)
    sc = acc.dynamic_scale_bytes_per_token(L, H)
    assert pay == g["fp8_payload_bytes_per_token"] and sc == g["dynamic_scale_bytes_per_token"]
    assert (pay + sc) / KiB == g["total_kib_per_token"]
    bf = acc.payload_bytes_per_token(L, H, D, 2)
    assert bf / KiB == g["bf16_kib_per_token"]
    assert round(bf / (pay + sc), 2) == g["compression_approx"]
    assert pay * T / GiB == g["fp8_data_gib"] and sc * T / MiB == g["scales_mib"]
    assert (pay + sc) * T / GiB == g["total_gib"] and bf * T / GiB == g["bf16_gib"]
    assert acc.block_bytes(pay + sc, bs) / KiB == g["block_kib"]


@pytest.mark.parametrize("D", [64, 128, 256])
def test_fp8_scale_tax(D):
    assert acc.fp8_scale_tax(D) * 100 == GOLD["scale_tax"]["fp8_percent"][str(D)]
    # the tax is metadata / payload whatever the layer and head counts
    assert acc.dynamic_scale_bytes_per_token(7, 3) / acc.payload_bytes_per_token(7, 3, D, 1) \
        == acc.fp8_scale_tax(D)


@pytest.mark.parametrize("D", [64, 128])
def test_int4_scale_tax(D):
    assert acc.int4_scale_tax(D) * 100 == GOLD["scale_tax"]["int4_percent"][str(D)]
    assert acc.dynamic_scale_bytes_per_token(5, 2) / acc.payload_bytes_per_token(5, 2, D, 0.5) \
        == acc.int4_scale_tax(D)


def test_static_per_head_with_q():
    g = GOLD["static_per_head_with_q"]
    assert acc.static_per_head_scale_count_with_q(g["q_heads"], g["kv_heads"]) == g["scale_count"]
    assert 4 * g["scale_count"] == g["bytes_per_layer"]
    extra = acc.static_per_head_extra_bytes_with_q(g["q_heads"], g["kv_heads"])
    assert extra == g["extra_bytes_per_layer"]
    assert extra * g["layers"] == g["extra_bytes_24_layers"]


def test_gpt_oss_skip_example():
    g = GOLD["gpt_oss_20b_skip"]
    windows = [g["window"], 0] * (g["layers"] // 2)
    skipped = [w > 0 for w in windows]
    r = acc.skip_accounting(g["context"], windows, skipped, g["kv_heads"], g["head_size"])
    assert r["A"] == g["A"] and r["S"] == g["S"]
    assert 12 * g["context"] == g["full_layer_positions"] and 12 * 128 == g["local_layer_positions"]
    assert 2 * r["C"] == g["bf16_bytes_per_position"]
    assert round(r["bf16_bytes"] / MiB) == g["bf16_mib_approx"]
    assert r["fp8_bytes"] / MiB == g["fp8_mib_approx"]
    assert round(r["mixed_bytes"] / MiB) == g["mixed_mib_approx"]
    assert (r["mixed_bytes"] - r["fp8_bytes"]) / MiB == g["mixed_minus_fp8_mib"]
    assert round(r["compression"], 3) == g["compression_approx"]


def test_equal_retention_half_skipped():
    r = acc.skip_accounting(4096, [0] * 8, [True, False] * 4, 8, 128)
    assert round(r["compression"], 2) == GOLD["equal_retention_half_skipped"]["compression_approx"]
