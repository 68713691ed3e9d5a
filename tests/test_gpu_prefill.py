"""GPU prefill attention against the oracle's prefill (each new token's
query attends causally, within the window, to the cache), with the decode
tolerance (tests/helpers.attention_tolerance) per output row.  Cases: the
workloads' shapes at sizes the oracle finishes in seconds, every mode, window
and full layers, several query tiles per sequence with ragged tails, empty
chunks, a whole sequence prefilled from position 0."""
import types

import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun
from tests.helpers import bits, check_attention

pytestmark = pytest.mark.gpu

MODES = [orc.FP8_PER_TOKEN_HEAD, orc.FP8_PER_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16,
         orc.FP8_PER_TENSOR]


def _wl(base, contexts):
    return wl.Workload(**{**base.__dict__, "context_lens": tuple(contexts)})


CASES = {
    # name: (workload, new tokens per sequence)
    "tiny": (wl.CONFIGS["tiny"], (37, 60)),
    "llama8b": (_wl(wl.CONFIGS["llama8b"], (600, 900, 1000)), (0, 150, 300)),
    "gptoss": (_wl(wl.CONFIGS["gptoss20b"], (700, 300, 129)), (150, 1, 129)),
    "gemma": (_wl(wl.CONFIGS["gemma_d256"], (1200, 700)), (300, 257)),
}


def _queries(w, T, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(T, w.Hq, w.D, generator=g).to(torch.bfloat16).cuda()


def _run(r, chunks, seed=11, max_query_len=None):
    kvq = K()
    w = r.w
    T = sum(chunks)
    q = _queries(w, T, seed)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32, device="cuda")
    out = torch.full((max(T, 1), w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    mq = max(chunks) if max_query_len is None else max_query_len
    kvq.kvq_prefill_attention(r.ctx, r.layer, q, r.kc, r.vc, r.pg.block_table, qs,
                              r.pg.context_lens, out, max_query_len=mq, k_scale=r.k_scale,
                              v_scale=r.v_scale, k_cache_scale=r.ks, v_cache_scale=r.vs)
    torch.cuda.synchronize()
    return q, qs, out


def _check(r, q, qs, out, pairs, where):
    kc, vc, ks, vs = r.host
    w = r.w
    bt = r.pg.block_table.cpu().numpy()
    qsn = qs.cpu().numpy()
    cl = r.pg.context_lens.cpu().numpy()
    ref = orc.prefill(r.mode, bits(q), kc, vc, bt, qsn, cl, k_scale=r.o_k_scale,
                      v_scale=r.o_v_scale, k_cache_scale=ks, v_cache_scale=vs, window=r.window,
                      block_size=w.block_size, pairs=pairs)
    # tolerance rows: each token is its own decode query with context p + 1
    seq = np.zeros(int(qsn[-1]), dtype=np.int64)
    ctx = np.zeros(int(qsn[-1]), dtype=np.int32)
    for b in range(len(cl)):
        n = int(qsn[b + 1] - qsn[b])
        seq[qsn[b]:qsn[b + 1]] = b
        ctx[qsn[b]:qsn[b + 1]] = int(cl[b]) - n + 1 + np.arange(n)
    view = types.SimpleNamespace(host=r.host, w=w, q=q, window=r.window, mode=r.mode,
                                 o_k_scale=r.o_k_scale, o_v_scale=r.o_v_scale,
                                 cl=torch.from_numpy(ctx),
                                 pg=types.SimpleNamespace(block_table=torch.from_numpy(bt[seq])))
    tol = LayerRun.tolerance(view, ref, pairs)
    got = out.cpu().numpy()[[p[0] for p in pairs], [p[1] for p in pairs]]
    check_attention(got, ref, tol, where)


def _pairs(T, Hq, limit=6000, seed=3):
    allp = [(t, h) for t in range(T) for h in range(Hq)]
    if len(allp) <= limit:
        return allp
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(len(allp), size=limit, replace=False))
    return [allp[i] for i in idx]


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("mode", MODES)
def test_prefill_matches_oracle(name, mode):
    w, chunks = CASES[name]
    kvq = K()
    for layer in sorted(set([0, w.num_layers - 1])):     # window layer and full layer
        r = LayerRun(w, mode, layer=layer)
        r.write()
        q, qs, out = _run(r, chunks)
        assert kvq.kvq_get_device_error() == 0
        _check(r, q, qs, out, _pairs(sum(chunks), w.Hq),
               f"{name} mode {mode} layer {layer} window {r.window}")


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD])
def test_whole_sequences_prefilled_from_position_zero(mode):
    w = _wl(wl.CONFIGS["llama8b"], (200, 333))
    r = LayerRun(w, mode)
    r.write()
    q, qs, out = _run(r, (200, 333), seed=12, max_query_len=400)
    assert K().kvq_get_device_error() == 0
    _check(r, q, qs, out, _pairs(533, w.Hq), f"from zero mode {mode}")


def test_chunk_longer_than_context_is_reported():
    w = wl.CONFIGS["tiny"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    kvq = K()
    q = _queries(w, 40, 13)
    qs = torch.tensor([0, 38, 40], dtype=torch.int32, device="cuda")   # 38 > context 37
    out = torch.zeros(40, w.Hq, w.D, device="cuda")
    kvq.kvq_prefill_attention(r.ctx, 0, q, r.kc, r.vc, r.pg.block_table, qs, r.pg.context_lens,
                              out, max_query_len=38, k_cache_scale=r.ks, v_cache_scale=r.vs)
    assert kvq.kvq_get_device_error() == kvq.STATUS.index("KVQ_ERR_BAD_INDEX")


@pytest.mark.parametrize("name,mode", [("llama8b", orc.FP8_PER_TOKEN_HEAD),
                                       ("llama8b", orc.INT4_PER_TOKEN_HEAD),
                                       ("llama8b", orc.BF16),
                                       ("gemma", orc.FP8_PER_TOKEN_HEAD)])
def test_bad_block_id_is_reported_and_masked(name, mode):
    """A block id past the cache in the middle of a sequence's table row: the
    prefill kernels fetch nothing for that page, report BAD_INDEX, and treat
    its positions as masked, so every output stays finite."""
    w, chunks = CASES[name]
    r = LayerRun(w, mode, layer=w.num_layers - 1)
    r.write()
    kvq = K()
    b = 1
    bt = r.pg.block_table.clone()
    bt[b, 3] = r.pg.num_blocks + 5
    T = sum(chunks)
    q = _queries(w, T, 17)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32, device="cuda")
    out = torch.full((T, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    kvq.kvq_prefill_attention(r.ctx, r.layer, q, r.kc, r.vc, bt, qs, r.pg.context_lens, out,
                              max_query_len=max(chunks), k_scale=r.k_scale, v_scale=r.v_scale,
                              k_cache_scale=r.ks, v_cache_scale=r.vs)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == kvq.STATUS.index("KVQ_ERR_BAD_INDEX")
    assert torch.isfinite(out).all()
