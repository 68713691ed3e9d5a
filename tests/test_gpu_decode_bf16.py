"""bf16-output decode: every element is the round-to-nearest-even bf16 of the
fp32 decode of the same call (same inputs, same worker count), and lies within
the fp32 decode's bar (tests/helpers.attention_tolerance) plus one bf16 unit
in the last place of the float64 oracle.  Cases cover the direct store of
single-worker items, the merge of split items, zero rows of empty contexts,
and the INT4 epilogue scaling."""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": wl.CONFIGS["tiny"],
    "llama8b": wl.scaled(wl.CONFIGS["llama8b"], batch=3, context=1000),
    "gemma": wl.scaled(wl.CONFIGS["gemma_d256"], batch=2, context=1200),
    "ragged": wl.Workload("ragged", Hq=32, Hkv=8, D=128, block_size=16,
                          context_lens=(0, 1, 17, 250, 1000), head_mult_loguniform=(0.5, 32.0),
                          outlier_p=0.01, outlier_factor=8.0, seed=78),
}


def _decode_both(r, workers):
    kvq = K()
    w = r.w
    q = wl.queries(w, r.device, layer=r.layer)
    cl = r.pg.context_lens
    max_ctx = int(cl.max().item())
    n, ws_bytes = kvq.kvq_decode_plan(r.ctx, r.layer, w.B, max_ctx, workers)
    ws = torch.full((max(ws_bytes, 16) // 4,), float("nan"), dtype=torch.float32,
                    device=r.device)
    args = dict(max_context=max_ctx, k_scale=r.k_scale, v_scale=r.v_scale,
                k_cache_scale=r.ks, v_cache_scale=r.vs, num_workers=n, workspace=ws)
    out32 = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device=r.device)
    kvq.kvq_decode_attention(r.ctx, r.layer, q, r.kc, r.vc, r.pg.block_table, cl, out32, **args)
    out16 = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=r.device)
    kvq.kvq_decode_attention_bf16(r.ctx, r.layer, q, r.kc, r.vc, r.pg.block_table, cl, out16,
                                  **args)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    return out32, out16, n


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16,
                                  orc.FP8_PER_HEAD])
@pytest.mark.parametrize("workers", [1, 7, 0])
def test_bf16_output_is_rounded_fp32_output(name, mode, workers):
    w = CASES[name]
    layer = w.num_layers - 1
    r = LayerRun(w, mode, layer=layer)
    r.write()
    out32, out16, n = _decode_both(r, workers)
    want = out32.to(torch.bfloat16)
    assert not torch.isnan(out32).any()
    same = out16.view(torch.int16) == want.view(torch.int16)
    assert bool(same.all()), (f"{name} mode {mode} workers {n}: "
                              f"{int((~same).sum())} of {same.numel()} bf16 outputs differ")
    # against the oracle: |bf16 out - oracle| <= tolerance + one bf16 ulp of the oracle
    r.q, r.cl = wl.queries(w, r.device, layer=r.layer), r.pg.context_lens
    pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    ref = r.oracle_decode(pairs)
    tol = r.tolerance(ref, pairs)
    got = out16.float().cpu().numpy().reshape(-1, w.D).astype(np.float64)
    mag = np.abs(ref)
    ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.maximum(mag, 1e-300))) - 7), 2.0 ** -133)
    err = np.abs(got - ref)
    assert np.all(err <= tol + ulp), (f"{name} mode {mode} workers {n}: worst bf16 error "
                                      f"{err.max():.3e} against the oracle")
