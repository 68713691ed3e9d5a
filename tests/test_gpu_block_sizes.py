"""Pages larger than 16 positions (block sizes 32, 64, 128): several 16-position
tiles per page for the decode, 64-key tiles inside or across pages for the
prefill, and the write's slot arithmetic; all against the oracle."""
import pytest

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun
from tests.test_gpu_prefill import _check, _pairs, _run

pytestmark = pytest.mark.gpu


def _w(bs, window=0):
    return wl.Workload(f"bs{bs}", Hq=8, Hkv=2, D=128, block_size=bs,
                       context_lens=(37, 300, 129, 0, 1000), windows=(window,),
                       head_mult=(1.0, 16.0), outlier_p=0.05, outlier_factor=4.0, seed=90 + bs)


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16])
@pytest.mark.parametrize("window", [0, 100])
def test_write_decode_prefill_with_larger_pages(bs, mode, window):
    w = _w(bs, window)
    r = LayerRun(w, mode)
    r.write()
    r.check_write()
    for workers in (1, 5, 0):
        out = r.decode(num_workers=workers)
        r.check_decode(out, where=f"bs {bs} mode {mode} window {window} workers {r.workers}")
    chunks = (37, 80, 129, 0, 300)
    q, qs, out = _run(r, chunks, seed=21)
    assert K().kvq_get_device_error() == 0
    _check(r, q, qs, out, _pairs(sum(chunks), w.Hq), f"prefill bs {bs} mode {mode} window {window}")
