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
def test_ragged_and_empty_contexts(mode, window):
    base = SMALL["llama8b"]
    w = wl.Workload("ragged", Hq=32, Hkv=8, D=128, block_size=16,
                    context_lens=(0, 1, 15, 16, 17, 33, 250, 1000), windows=(window,),
                    head_mult_loguniform=(0.5, 32.0), outlier_p=0.01, outlier_factor=8.0,
                    seed=77)
    r = LayerRun(w, mode)
    r.write()
    for workers in (1, 4, 13, 0):
        out = r.decode(num_workers=workers)
        assert torch.all(out[0] == 0), "empty context must give zeros"
        r.check_decode(out, where=f"ragged w{window} workers {workers}")


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
