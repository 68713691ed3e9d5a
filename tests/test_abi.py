"""The C ABI without a GPU: the library loads, exports every declared entry
point, validates arguments on the host, and its capacity accounting matches
the pages' formulas (oracle/accounting.py) and printed numbers."""
import ctypes
import json
import os
import re

import pytest

from oracle import accounting as acc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "accounting.json")))

kvq = pytest.importorskip("int4_quantized_paged_gb300.kvq",
                          reason="libkvq.so not built (run __graft_entry__.build())")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def _ctx(modes, windows=None, Hq=32, Hkv=8, D=128, bs=16, nb=64):
    return kvq.kvq_create(len(modes), Hq, Hkv, D, bs, nb, modes, windows)


def test_create_validates_config():
    with pytest.raises(kvq.KVQError, match="UNSUPPORTED"):
        _ctx([3], D=96)
    with pytest.raises(kvq.KVQError, match="UNSUPPORTED"):
        _ctx([3], bs=24)
    with pytest.raises(kvq.KVQError, match="INVALID_ARG"):
        _ctx([3], Hq=30)
    with pytest.raises(kvq.KVQError, match="INVALID_ARG"):
        _ctx([7])
    with pytest.raises(kvq.KVQError, match="INVALID_ARG"):
        _ctx([3], windows=[-1])
    with pytest.raises(kvq.KVQError, match="UNSUPPORTED"):
        _ctx([3], Hq=96, Hkv=4)      # GQA ratio 24 not built
    # a BF16 D=256 layer of 2^30 cells spans 2^32 rows of 128 bytes: past the
    # signed 32-bit TMA coordinate; the same pool in FP8 D=128 spans 2^30
    with pytest.raises(kvq.KVQError, match="UNSUPPORTED"):
        _ctx([0], Hq=16, Hkv=8, D=256, nb=1 << 23)
    _ctx([3], Hq=16, Hkv=8, D=128, nb=1 << 23)


def test_layer_buffer_sizes():
    ctx = _ctx([0, 1, 2, 3, 4], nb=10)
    cells = 10 * 8 * 16
    assert kvq.kvq_layer_buffer_sizes(ctx, 0) == (cells * 256, 0)
    assert kvq.kvq_layer_buffer_sizes(ctx, 1) == (cells * 128, 0)
    assert kvq.kvq_layer_buffer_sizes(ctx, 2) == (cells * 128, 0)
    assert kvq.kvq_layer_buffer_sizes(ctx, 3) == (cells * 128, cells * 4)
    assert kvq.kvq_layer_buffer_sizes(ctx, 4) == (cells * 64, cells * 4)
    with pytest.raises(kvq.KVQError):
        kvq.kvq_layer_buffer_sizes(ctx, 5)


def test_capacity_32_layer_example():
    g = GOLD["gqa_32_layer"]
    ctx = _ctx([3] * g["layers"], Hq=32, Hkv=g["kv_heads"], D=g["head_size"])
    r = kvq.kvq_cache_bytes(ctx, g["context"])
    assert r["payload_bytes_per_token"] == acc.payload_bytes_per_token(32, 8, 128, 1)
    assert r["scale_bytes_per_token"] == acc.dynamic_scale_bytes_per_token(32, 8)
    assert r["bytes_per_token"] / 1024 == g["total_kib_per_token"]
    assert r["block_bytes"] / 1024 == g["block_kib"]
    assert r["cache_bytes"] / 2 ** 30 == g["total_gib"]
    assert r["bf16_cache_bytes"] / 2 ** 30 == g["bf16_gib"]


def test_capacity_80_layer_static_metadata():
    g = GOLD["fp8_80_layer_128k"]
    for mode, key in ((1, "per_tensor_metadata_bytes"), (2, "static_per_head_metadata_bytes")):
        ctx = _ctx([mode] * 80)
        r = kvq.kvq_cache_bytes(ctx, g["context"])
        assert r["static_scale_bytes"] == g[key]
        assert r["cache_bytes"] - r["static_scale_bytes"] == g["fp8_kv_bytes"]
    ctx = _ctx([3] * 80)
    r = kvq.kvq_cache_bytes(ctx, g["context"])
    assert r["cache_bytes"] / 2 ** 30 == g["fp8_plus_scales_gib"]


def test_capacity_gpt_oss_skip_example():
    g = GOLD["gpt_oss_20b_skip"]
    wins = [128, 0] * 12
    ref = acc.skip_accounting(g["context"], wins, [w > 0 for w in wins], 8, 64)
    all_fp8 = kvq.kvq_cache_bytes(_ctx([1] * 24, wins, Hq=64, D=64), g["context"])
    mixed = kvq.kvq_cache_bytes(_ctx([0, 1] * 12, wins, Hq=64, D=64), g["context"])
    assert all_fp8["retained_positions"] == ref["A"]
    assert all_fp8["cache_bytes"] - all_fp8["static_scale_bytes"] == ref["fp8_bytes"]
    assert mixed["cache_bytes"] - mixed["static_scale_bytes"] == ref["mixed_bytes"]
    assert all_fp8["bf16_cache_bytes"] == ref["bf16_bytes"]


def test_write_rejects_bad_arguments_without_launching():
    ctx = _ctx([3, 1])
    ok = 0x10000000                       # never dereferenced: validation fails first
    args = dict(k_new=ok, v_new=ok, slot_mapping=ok, k_cache=ok, v_cache=ok,
                k_cache_scale=ok, v_cache_scale=ok)
    L = kvq._lib

    def write(layer=0, T=4, stride=0, **over):
        a = dict(args, **over)
        return L.kvq_cache_write(ctx, layer, a["k_new"], a["v_new"], stride, a["slot_mapping"],
                                 T, a.get("k_scale"), a.get("v_scale"), a["k_cache"],
                                 a["v_cache"], a["k_cache_scale"], a["v_cache_scale"], None)
    assert write(T=0) == 0
    assert write(T=-1) == 1
    assert write(layer=2) == 1
    assert write(k_new=None) == 1
    assert write(k_cache_scale=None) == 1
    assert write(layer=1) == 1                   # per-tensor needs k_scale / v_scale
    assert write(k_new=ok + 8) == 3
    assert write(k_cache=ok + 4) == 3
    assert write(stride=8 * 128 + 4) == 3
    assert write(stride=100) == 1


def test_decode_plan_and_workspace_rules():
    ctx = _ctx([3], Hq=64, Hkv=8, D=128)
    w, ws = kvq.kvq_decode_plan(ctx, 0, 8, 131072)
    assert w >= 1 and ws == (0 if w == 1 else (8 * 8 + w) * 8 * 130 * 4 + (8 * 8 + 1) * 8)
    w1, ws1 = kvq.kvq_decode_plan(ctx, 0, 8, 131072, num_workers=1)
    assert (w1, ws1) == (1, 0)
    w5, ws5 = kvq.kvq_decode_plan(ctx, 0, 8, 131072, num_workers=5)
    assert (w5, ws5) == (5, (8 * 8 + 5) * 8 * 130 * 4 + (8 * 8 + 1) * 8)
    # a short context never gets more workers than it has 64-position chunks
    ws_small, _ = kvq.kvq_decode_plan(ctx, 0, 1, 64)
    assert ws_small <= 8 * 2
    ok = 0x10000000
    L = kvq._lib
    # too-small workspace is refused before launch
    rc = L.kvq_decode_attention(ctx, 0, ok, ok, ok, None, None, ok, ok, ok, 8192, ok, 8, 131072,
                                ok, 5, ok, ws5 - 1, None)
    assert rc == 4
    rc = L.kvq_decode_attention(ctx, 0, ok + 2, ok, ok, None, None, ok, ok, ok, 8192, ok, 8,
                                131072, ok, 1, None, 0, None)
    assert rc == 3
    rc = L.kvq_decode_attention(ctx, 0, ok, ok, ok, None, None, None, ok, ok, 8192, ok, 8,
                                131072, ok, 1, None, 0, None)
    assert rc == 1
    assert L.kvq_decode_attention(ctx, 0, ok, ok, ok, None, None, ok, ok, ok, 8192, ok, 0,
                                  0, ok, 1, None, 0, None) == 0


def test_workspace_size_is_the_automatic_plan():
    ctx = _ctx([3, 0], windows=[0, 128], Hq=64, Hkv=8, D=128)
    for layer, batch, ctxlen in ((0, 8, 131072), (0, 1, 64), (1, 16, 32768), (0, 0, 0)):
        assert kvq.kvq_decode_workspace_size(ctx, layer, batch, ctxlen) == \
            kvq.kvq_decode_plan(ctx, layer, batch, ctxlen)[1]
    assert kvq.kvq_decode_workspace_size(ctx, 2, 8, 4096) == 0      # no such layer
    assert kvq.kvq_decode_workspace_size(ctx, 0, -1, 4096) == 0     # invalid batch


def test_bf16_output_decode_validates_like_fp32():
    ctx = _ctx([3], Hq=64, Hkv=8, D=128)
    _, ws5 = kvq.kvq_decode_plan(ctx, 0, 8, 131072, num_workers=5)
    ok = 0x10000000
    L = kvq._lib
    f = L.kvq_decode_attention_bf16
    assert f(ctx, 0, ok, ok, ok, None, None, ok, ok, ok, 8192, ok, 8, 131072, ok, 5, ok,
             ws5 - 1, None) == 4                                 # workspace too small
    assert f(ctx, 0, ok, ok, ok, None, None, ok, ok, ok, 8192, ok, 8, 131072, ok + 8, 1, None,
             0, None) == 3                                        # output not 16-byte aligned
    assert f(ctx, 0, ok, ok, ok, None, None, ok, ok, ok, 8192, ok, 8, 131072, None, 1, None, 0,
             None) == 1                                           # no output
    assert f(ctx, 0, ok, ok, ok, None, None, ok, ok, ok, 8192, ok, 0, 0, ok, 1, None, 0,
             None) == 0                                           # empty batch


def test_status_strings():
    for s in range(8):
        assert kvq.kvq_status_string(s)


def test_header_is_plain_c_and_links(tmp_path):
    """include/kvq.h compiles as C99 with warnings as errors, and a C program
    using only host-side calls links against libkvq.so and runs."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(kvq.LIB_PATH)
    lib_name = os.path.basename(kvq.LIB_PATH)
    src = tmp_path / "use_kvq.c"
    src.write_text(r'''
#include <stdio.h>
#include "kvq.h"
int main(void) {
  int modes[2] = {KVQ_FP8_PER_TOKEN_HEAD, KVQ_BF16};
  int windows[2] = {0, 128};
  kvq_config cfg = {2, 32, 8, 128, 16, 1024, modes, windows, 0.0f};
  kvq_ctx* ctx = NULL;
  kvq_status st = kvq_create(&cfg, &ctx);
  if (st != KVQ_OK) { printf("create: %s\n", kvq_status_string(st)); return 1; }
  size_t code = 0, scale = 0;
  st = kvq_layer_buffer_sizes(ctx, 0, &code, &scale);
  printf("%d %zu %zu\n", (int)st, code, scale);
  kvq_destroy(ctx);
  return st == KVQ_OK && code == 1024u * 8u * 16u * 128u && scale == 1024u * 8u * 16u * 4u ? 0 : 2;
}
''')
    exe = tmp_path / "use_kvq"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(ROOT, "include"), str(src), "-L", lib_dir, "-l:" + lib_name,
                        "-Wl,-rpath," + lib_dir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_fp8_query_without_scale_is_an_argument_error():
    ctx = _ctx([3], Hq=64, Hkv=8, D=128)
    ok = 0x10000000
    with pytest.raises(kvq.KVQError, match="INVALID_ARG"):
        kvq.kvq_decode_attention_fp8_query(ctx, 0, ok, None, ok, ok, ok, ok, ok, max_context=4096,
                                           k_cache_scale=ok, v_cache_scale=ok, batch=8,
                                           max_blocks_per_seq=256, stream=0)
