"""FP8-query decode on the GPU against the oracle's FP8-query decode
(q_hat = E4M3(RN32(q / s)) x s, one scale or one per query head), with the
tolerance of test_gpu_decode.py."""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun, sample_pairs
from tests.helpers import bits, check_attention

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": wl.CONFIGS["tiny"],
    "llama8b": wl.scaled(wl.CONFIGS["llama8b"], batch=3, context=1000),
    "gptoss": wl.scaled(wl.CONFIGS["gptoss20b"], batch=2, context=500),
    "gemma": wl.scaled(wl.CONFIGS["gemma_d256"], batch=2, context=1200),
}


def _scales(w, per_head):
    if not per_head:
        return np.array([0.02], dtype=np.float32)
    return np.exp(np.linspace(np.log(0.005), np.log(0.5), w.Hq)).astype(np.float32)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.FP8_PER_HEAD,
                                  orc.INT4_PER_TOKEN_HEAD, orc.BF16])
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("workers", [1, 0])
def test_fp8_query_decode_matches_oracle(name, mode, per_head, workers):
    kvq = K()
    w = CASES[name]
    layer = w.num_layers - 1
    r = LayerRun(w, mode, layer=layer)
    r.write()
    q = wl.queries(w, r.device, layer=layer)
    qs_host = _scales(w, per_head)
    qs = torch.tensor(qs_host, device=r.device)
    cl = r.pg.context_lens
    max_ctx = int(cl.max().item())
    n, ws_bytes = kvq.kvq_decode_plan(r.ctx, layer, w.B, max_ctx, workers)
    ws = torch.full((max(ws_bytes, 16) // 4,), float("nan"), dtype=torch.float32,
                    device=r.device)
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device=r.device)
    kvq.kvq_decode_attention_fp8_query(r.ctx, layer, q, qs, r.kc, r.vc, r.pg.block_table, cl,
                                       out, max_context=max_ctx, k_scale=r.k_scale,
                                       v_scale=r.v_scale, k_cache_scale=r.ks,
                                       v_cache_scale=r.vs, num_workers=n, workspace=ws)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    r.q, r.cl = q, cl
    pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    kc, vc, ks, vs = r.host
    ref = orc.decode_fp8_query(mode, bits(q), qs_host, kc, vc, r.pg.block_table.cpu().numpy(),
                               cl.cpu().numpy(), k_scale=r.o_k_scale, v_scale=r.o_v_scale,
                               k_cache_scale=ks, v_cache_scale=vs, window=r.window,
                               block_size=w.block_size, pairs=pairs)
    got = out.cpu().numpy()[[p[0] for p in pairs], [p[1] for p in pairs]]
    check_attention(got, ref, r.tolerance(ref, pairs),
                    f"{name} mode {mode} per_head {per_head} workers {n}")


def test_fp8_query_rejects_bad_scale_count():
    kvq = K()
    w = CASES["tiny"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    q = wl.queries(w, r.device)
    out = torch.empty(w.B, w.Hq, w.D, device=r.device)
    with pytest.raises(kvq.KVQError, match="INVALID_ARG"):
        kvq.kvq_decode_attention_fp8_query(r.ctx, 0, q, torch.ones(3, device=r.device), r.kc,
                                           r.vc, r.pg.block_table, r.pg.context_lens, out,
                                           max_context=100, k_cache_scale=r.ks,
                                           v_cache_scale=r.vs, num_workers=1)
