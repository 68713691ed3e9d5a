"""Prefill at the group sizes the workloads do not use, on both prefill
kernels' shapes: G = 1 (a query tile of 128 positions, so the two query tiles
of one CTA span 256 positions, wider than a 100-token window) and G = 2, at
head_dim 64, 128 and 256 (one query tile per CTA, Q in tensor memory), window
and full layers, quantized modes (the
warp-specialised kernel) and BF16 (the single-role kernel), with ragged
chunks that leave the second query tile of the last CTA partly or wholly
empty.  Each output row is checked against the oracle's prefill with the
decode tolerance, checked as the decode of that query."""
import pytest

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun
from tests.test_gpu_prefill import _check, _pairs, _run

pytestmark = pytest.mark.gpu

SHAPES = {
    # name: (Hq, Hkv, D, context lens, new tokens per sequence)
    "g1-d128": (8, 8, 128, (700, 333, 300), (300, 77, 256)),
    "g2-d64": (8, 4, 64, (650, 129), (257, 129)),
    "g1-d64": (4, 4, 64, (520, 40), (400, 40)),
    "g1-d256": (4, 4, 256, (530, 300), (260, 300)),
}


def _workload(name):
    Hq, Hkv, D, ctx, _ = SHAPES[name]
    return wl.Workload(name, Hq=Hq, Hkv=Hkv, D=D, block_size=16, context_lens=ctx,
                       windows=(100, 0), head_mult_loguniform=(0.5, 8.0), outlier_p=0.01,
                       outlier_factor=4.0, seed=4321 + Hq + D)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD,
                                  orc.FP8_PER_HEAD, orc.BF16])
@pytest.mark.parametrize("layer", [0, 1])
def test_prefill_group_sizes(name, mode, layer):
    w = _workload(name)
    chunks = SHAPES[name][4]
    r = LayerRun(w, mode, layer=layer)
    r.write()
    q, qs, out = _run(r, chunks, seed=21 + layer)
    assert K().kvq_get_device_error() == 0
    _check(r, q, qs, out, _pairs(sum(chunks), w.Hq),
           f"{name} mode {mode} layer {layer} window {r.window}")
