"""One cache whose layers differ in mode and window, run as the decode step.

The layer-skipping recipe of "FP8 KV cache layer skipping vs per-head
scales" (opening section; "Layer skipping follows retained-token
footprint") keeps the sliding-window layers in BF16 and quantizes the full
layers.  Here one kvq_ctx holds such layers (scaled down from the
gpt-oss-20b-like workload: Hq 64, Hkv 8, D 64, windows alternating 128 and
full) plus a second mix of all quantized modes.  Each layer's cache is filled
with the context minus the current token; then the decode step writes the
current token and decodes, layer after layer on one stream with no sync in
between, eagerly and replayed as a CUDA graph.  Every layer is compared with
the oracle, so a dispatch that took any layer's mode or window from another
layer fails.
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun
from tests.helpers import bits

pytestmark = pytest.mark.gpu

BASE = wl.scaled(wl.CONFIGS["gptoss20b"], batch=3, context=700)

MIXES = {
    # the skip variant: window layers BF16, full layers dynamic FP8
    "skip_sliding": ([orc.BF16, orc.FP8_PER_TOKEN_HEAD] * 2, (128, 0, 128, 0)),
    # every mode once, windows of different lengths
    "all_modes": ([orc.FP8_PER_TOKEN_HEAD, orc.BF16, orc.INT4_PER_TOKEN_HEAD, orc.FP8_PER_HEAD,
                   orc.FP8_PER_TENSOR], (128, 0, 40, 0, 300)),
}


@pytest.mark.parametrize("mix", list(MIXES))
def test_mixed_layer_modes_decode_step(mix):
    kvq = K()
    modes, windows = MIXES[mix]
    w = wl.Workload(**{**BASE.__dict__, "windows": windows})
    L = w.context_lens[0]
    runs = []
    for li, mode in enumerate(modes):
        r = LayerRun(w, mode, layer=li)
        runs.append(r)
    # one context for every layer (the per-layer runs only supply inputs and
    # the oracle side)
    ctx = kvq.kvq_create(w.num_layers, w.Hq, w.Hkv, w.D, w.block_size, runs[0].pg.num_blocks,
                         modes, list(windows))
    for r in runs:
        r.ctx = ctx
        r.kc, r.vc, r.ks, r.vs = kvq.alloc_layer_cache(ctx, r.layer, "cuda")
        r.write([torch.arange(0, L - 1) for _ in range(w.B)])   # all but the current token
    pg = runs[0].pg
    slots = wl.slot_mapping(w, pg, [torch.tensor([L - 1]) for _ in range(w.B)], "cuda")
    step_in = []
    for r in runs:
        k_new, v_new = wl.kv_tokens(w, w.B, "cuda", layer=r.layer, stream_base=700)
        q = wl.queries(w, "cuda", layer=r.layer)
        workers, ws_bytes = kvq.kvq_decode_plan(ctx, r.layer, w.B, L, 0)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        step_in.append((k_new, v_new, q, workers, ws, out))
        # the oracle writes the same current token
        kc, vc, ks, vs = r.host
        orc.cache_write(r.mode, bits(k_new), bits(v_new), slots.cpu().numpy(), kc, vc, ks, vs,
                        k_scale=r.o_k_scale, v_scale=r.o_v_scale)

    def step():
        for r, (k_new, v_new, q, workers, ws, out) in zip(runs, step_in):
            kvq.kvq_cache_write(ctx, r.layer, k_new, v_new, slots, r.kc, r.vc, r.ks, r.vs,
                                r.k_scale, r.v_scale)
            kvq.kvq_decode_attention(ctx, r.layer, q, r.kc, r.vc, pg.block_table,
                                     pg.context_lens, out, max_context=L, k_scale=r.k_scale,
                                     v_scale=r.v_scale, k_cache_scale=r.ks, v_cache_scale=r.vs,
                                     num_workers=workers, workspace=ws)

    step()
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    eager = [s[5].clone() for s in step_in]
    for r, (k_new, v_new, q, workers, ws, out) in zip(runs, step_in):
        r.check_write()
        r.q, r.cl = q, pg.context_lens
        r.check_decode(out, where=f"{mix} layer {r.layer} mode {r.mode} window {r.window}")

    # the same step replayed as a CUDA graph (re-writing the current token is
    # idempotent): identical outputs
    for s in step_in:
        s[5].fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    for li, s in enumerate(step_in):
        assert torch.equal(s[5].view(torch.int32), eager[li].view(torch.int32)), \
            f"{mix} layer {li}: graph replay differs from the eager step"
