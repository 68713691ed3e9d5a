"""GPU decode attention against the float64 oracle.

Bar: relative L2 <= 1e-3 over each output tensor, and every element within
2e-3 plus the fp32 forward-error term of tests/helpers.attention_tolerance
(which is 2e-3 for heads whose values are O(1)).  Cases: the five workloads
scaled to sizes the oracle finishes in seconds, every mode, forced and
automatic split counts, windows, ragged and empty contexts; and the full
benchmark sizes on sampled (sequence, head) rows.
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun, sample_pairs
from tests.helpers import bits

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": wl.CONFIGS["tiny"],
    "llama8b": wl.scaled(wl.CONFIGS["llama8b"], batch=3, context=1000),
    "llama70b": wl.scaled(wl.CONFIGS["llama70b_128k"], batch=2, context=2500),
    "gptoss": wl.scaled(wl.CONFIGS["gptoss20b"], batch=3, context=700),
    "gemma": wl.scaled(wl.CONFIGS["gemma_d256"], batch=2, context=1200),
}
ALL_MODES = [orc.BF16, orc.FP8_PER_TENSOR, orc.FP8_PER_HEAD, orc.FP8_PER_TOKEN_HEAD,
             orc.INT4_PER_TOKEN_HEAD]


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode", ALL_MODES)
@pytest.mark.parametrize("workers", [1, 3, 37, 0])
def test_decode_small(name, mode, workers):
    w = SMALL[name]
    for layer in sorted(set([0, w.num_layers - 1])):   # window layer and full layer
        r = LayerRun(w, mode, layer=layer)
        r.write()
        out = r.decode(num_workers=workers)
        r.check_decode(out, where=f"{name} mode {mode} layer {layer} workers {r.workers}")


def test_tiny_per_tensor_one_control():
    r = LayerRun(wl.CONFIGS["tiny"], orc.FP8_PER_TENSOR, per_tensor_scale=1.0)
    r.write()
    r.check_write()
    r.check_decode(r.decode())


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16])
@pytest.mark.parametrize("window", [0, 40])
@pytest.mark.parametrize("D", [128, 64])
def test_ragged_and_empty_contexts(mode, window, D):
    """Contexts that end inside a 16-position page tile, on its boundary and
    one past it, with and without a window (window starts inside a tile), at
    head_dim 128 and 64 (1 KB page tiles for FP8, 512 bytes for INT4), each
    with one, several and the automatic number of workers."""
    w = wl.Workload("ragged", Hq=32, Hkv=8, D=D, block_size=16,
                    context_lens=(0, 1, 15, 16, 17, 33, 250, 1000), windows=(window,),
                    head_mult_loguniform=(0.5, 32.0), outlier_p=0.01, outlier_factor=8.0,
                    seed=77)
    r = LayerRun(w, mode)
    r.write()
    for workers in (1, 4, 13, 0):
        out = r.decode(num_workers=workers)
        assert torch.all(out[0] == 0), "empty context must give zeros"
        r.check_decode(out, where=f"ragged D{D} w{window} workers {workers}")


def test_shorter_context_than_written_and_worker_independence():
    # context_lens below the written length: positions past L are never read.
    w = SMALL["llama70b"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    cl = torch.tensor([1234, 7], dtype=torch.int32, device="cuda")
    outs = [r.decode(num_workers=s, context_lens=cl) for s in (1, 2, 7, 100, 0)]
    for o in outs:
        r.check_decode(o)
    for o in outs[1:]:
        assert torch.allclose(o, outs[0], rtol=1e-4, atol=1e-4)


def test_bad_block_id_is_reported_and_skipped():
    w = SMALL["tiny"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    kvq = K()
    bt = r.pg.block_table.clone()
    bt[1, 2] = r.pg.num_blocks + 5
    out = torch.empty(w.B, w.Hq, w.D, device="cuda")
    kvq.kvq_decode_attention(r.ctx, 0, wl.queries(w, "cuda"), r.kc, r.vc, bt,
                             r.pg.context_lens, out, max_context=100, k_cache_scale=r.ks,
                             v_cache_scale=r.vs, num_workers=1)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == kvq.STATUS.index("KVQ_ERR_BAD_INDEX")
    assert torch.isfinite(out).all()


# ------------------------------------------------------------ full sizes
@pytest.mark.parametrize("mode", [orc.FP8_PER_TENSOR, orc.FP8_PER_HEAD, orc.FP8_PER_TOKEN_HEAD])
def test_llama8b_full_size_sampled(mode):
    w = wl.CONFIGS["llama8b"]
    r = LayerRun(w, mode)
    r.write()
    out = r.decode()                       # the benchmark's launch configuration
    r.check_decode(out, pairs=sample_pairs(w, 48, seed=mode))


@pytest.mark.parametrize("mode", [orc.FP8_PER_TENSOR, orc.FP8_PER_HEAD, orc.FP8_PER_TOKEN_HEAD])
def test_llama70b_128k_full_size_sampled(mode):
    w = wl.CONFIGS["llama70b_128k"]
    r = LayerRun(w, mode)
    r.write()
    out = r.decode()
    r.check_decode(out, pairs=sample_pairs(w, 12, seed=mode))


@pytest.mark.parametrize("skip_sliding", [False, True])
def test_gptoss_full_size_window_and_full_layer(skip_sliding):
    w = wl.CONFIGS["gptoss20b"]
    for layer in (0, 1):                   # W=128 layer, full layer
        mode = orc.BF16 if (skip_sliding and layer == 0) else orc.FP8_PER_TOKEN_HEAD
        r = LayerRun(w, mode, layer=layer)
        r.write()
        out = r.decode()
        r.check_decode(out, pairs=sample_pairs(w, 24, seed=layer))


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD])
def test_gemma_full_size_sampled(mode):
    w = wl.CONFIGS["gemma_d256"]
    for layer in (0, 1):
        r = LayerRun(w, mode, layer=layer)
        r.write()
        out = r.decode()
        r.check_decode(out, pairs=sample_pairs(w, 16, seed=layer))


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16])
def test_window_layer_ring_reuse_of_blocks(mode):
    """A window layer paged as a ring of ceil(W/bs)+1 blocks per sequence,
    filled with the retained positions and then advanced token by token
    (each write overwrites a dead block), decodes exactly like the same layer
    paged with one block per logical block, and matches the oracle."""
    window = 40
    base = wl.Workload("ring", Hq=32, Hkv=8, D=128, block_size=16,
                       context_lens=(70, 300, 41, 1000), windows=(window,),
                       head_mult_loguniform=(0.5, 32.0), outlier_p=0.01, outlier_factor=8.0,
                       seed=91)
    steps = 20
    final = wl.Workload(**{**base.__dict__,
                           "context_lens": tuple(L + steps for L in base.context_lens)})
    kvq = K()
    runs = {}
    for kind in ("ring", "flat"):
        r = LayerRun(final, mode)
        if kind == "ring":
            r.pg = wl.ring_paging(final, window, r.device)
            r.ctx = kvq.kvq_create(1, final.Hq, final.Hkv, final.D, final.block_size,
                                   r.pg.num_blocks, [mode], [window])
            r.kc, r.vc, r.ks, r.vs = kvq.alloc_layer_cache(r.ctx, 0, r.device)
        runs[kind] = r
    # identical token streams for both layouts: the retained positions of the
    # starting contexts, then `steps` single-token writes per sequence
    for r in runs.values():
        r.static_scales()
    T0 = sum(min(L, window) for L in base.context_lens)
    k0, v0 = wl.kv_tokens(final, T0, "cuda", stream_base=500)
    pos0 = [torch.arange(max(0, L - window), L) for L in base.context_lens]
    outs = {}
    for kind, r in runs.items():
        slots = wl.slot_mapping(final, r.pg, pos0, "cuda")
        kvq.kvq_cache_write(r.ctx, 0, k0, v0, slots, r.kc, r.vc, r.ks, r.vs, r.k_scale, r.v_scale)
    for s in range(steps):
        ks_, vs_ = wl.kv_tokens(final, final.B, "cuda", stream_base=600 + s)
        cl = torch.tensor([L + s + 1 for L in base.context_lens], dtype=torch.int32,
                          device="cuda")
        q = wl.queries(final, "cuda", layer=0)
        for kind, r in runs.items():
            slots = wl.slot_mapping(final, r.pg, [torch.tensor([L + s]) for L in base.context_lens],
                                    "cuda")
            kvq.kvq_cache_write(r.ctx, 0, ks_, vs_, slots, r.kc, r.vc, r.ks, r.vs,
                                r.k_scale, r.v_scale)
            out = r.decode(num_workers=0, context_lens=cl, q=q)
            outs[kind] = out
        assert torch.equal(outs["ring"].view(torch.int32), outs["flat"].view(torch.int32)), \
            f"step {s}: ring-paged decode differs from the flat layout"
    # the final state against the oracle, through the ring's own block table
    r = runs["ring"]
    kc, vc, ks, vs = orc.alloc_cache(mode, r.pg.num_blocks, final.Hkv, final.block_size, final.D)
    slots0 = wl.slot_mapping(final, r.pg, pos0, "cuda")
    orc.cache_write(mode, bits(k0), bits(v0), slots0.cpu().numpy(), kc, vc, ks, vs,
                    k_scale=r.o_k_scale, v_scale=r.o_v_scale)
    for s in range(steps):
        ks_, vs_ = wl.kv_tokens(final, final.B, "cuda", stream_base=600 + s)
        slots = wl.slot_mapping(final, r.pg, [torch.tensor([L + s]) for L in base.context_lens],
                                "cuda")
        orc.cache_write(mode, bits(ks_), bits(vs_), slots.cpu().numpy(), kc, vc, ks, vs,
                        k_scale=r.o_k_scale, v_scale=r.o_v_scale)
    r.host = (kc, vc, ks, vs)
    r.check_decode(outs["ring"], where=f"ring mode {mode}")


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.BF16])
@pytest.mark.parametrize("workers", [7, 0])
def test_batch_above_128_sequences(mode, workers):
    """More than 128 sequences: warps find their share by the two-pass scan
    rather than the single round of context-length loads."""
    rng = np.random.default_rng(17)
    lens = tuple(int(x) for x in rng.integers(0, 200, size=150))
    w = wl.Workload("wide", Hq=4, Hkv=2, D=64, block_size=16, context_lens=lens, windows=(0,),
                    head_mult=(1.0, 16.0), outlier_p=0.05, outlier_factor=4.0, seed=83)
    r = LayerRun(w, mode)
    r.write()
    out = r.decode(num_workers=workers)
    r.check_decode(out, where=f"wide batch mode {mode} workers {r.workers}")


@pytest.mark.parametrize("scale", [0.03, 2.5])
def test_per_tensor_scale_other_than_one(scale):
    """The per-tensor path with K and V scales that are not 1: the scale enters
    the write's division, the decode's score factor and its unscale."""
    w = SMALL["llama8b"]
    r = LayerRun(w, orc.FP8_PER_TENSOR, per_tensor_scale=scale)
    r.write()
    r.check_write()
    r.check_decode(r.decode(num_workers=0), where=f"per-tensor scale {scale}")


@pytest.mark.parametrize("workers", [1, 0])
def test_context_past_its_block_table_row_is_clamped_and_reported(workers):
    """A context length beyond the positions its block-table row covers is an
    index error: only the covered positions are read, the BAD_INDEX bit is
    set, and the other sequences are unaffected.  The table is the front of a
    larger buffer, so even a read past its last row would stay in allocated
    memory."""
    kvq = K()
    w = SMALL["llama8b"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    maxb = r.pg.max_blocks
    cap = maxb * w.block_size
    padded = torch.zeros(w.B * maxb + 64, dtype=torch.int32, device="cuda")
    padded[:w.B * maxb] = r.pg.block_table.reshape(-1)
    bt = padded[:w.B * maxb].view(w.B, maxb)
    cl = r.pg.context_lens.clone()
    cl[w.B - 1] = cap + 40
    q = wl.queries(w, "cuda")
    nw, ws_bytes = kvq.kvq_decode_plan(r.ctx, 0, w.B, cap, workers)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
    with pytest.raises(kvq.KVQError, match="INVALID_ARG"):      # the plan's bound is checked
        kvq.kvq_decode_attention(r.ctx, 0, q, r.kc, r.vc, bt, cl, out, max_context=cap + 1,
                                 k_cache_scale=r.ks, v_cache_scale=r.vs, num_workers=nw,
                                 workspace=ws)
    kvq.kvq_decode_attention(r.ctx, 0, q, r.kc, r.vc, bt, cl, out, max_context=cap,
                             k_cache_scale=r.ks, v_cache_scale=r.vs, num_workers=nw, workspace=ws)
    torch.cuda.synchronize()
    assert kvq.STATUS[kvq.kvq_get_device_error()] == "KVQ_ERR_BAD_INDEX"
    assert torch.isfinite(out).all()
    r.q, r.cl = q, cl.clamp(max=cap)
    r.check_decode(out, where=f"context past its table row, workers {nw}")
