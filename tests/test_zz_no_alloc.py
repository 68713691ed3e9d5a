"""The allocation-free decode entry point (kvq_decode_attention_fixed_scratch).

Some callers cannot hand the library a device workspace: a serving loop that
forbids device allocations once it has started, a plugin inside a process
whose host owns every device buffer, or a binding with no device allocator.
For them the library keeps its split-K partials in one static device array.
This file checks, through the C ABI, that the entry point gives the same
attention output as kvq_decode_attention with a caller workspace, on two calls
in a row (the array keeps the previous call's contents), and that a request
too large for the array is refused before anything is launched.  It is
collected last so that a failure here never hides another test's result.
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun, sample_pairs
from tests.helpers import check_attention

pytestmark = pytest.mark.gpu


def _fixed(r, out, workers):
    kvq = K()
    w = r.w
    kvq.kvq_decode_attention_fixed_scratch(
        r.ctx, r.layer, r.q, r.kc, r.vc, r.pg.block_table, r.pg.context_lens, out,
        max_context=int(r.pg.context_lens.max()), k_scale=r.k_scale, v_scale=r.v_scale,
        k_cache_scale=r.ks, v_cache_scale=r.vs, num_workers=workers)


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD, orc.BF16])
def test_fixed_scratch_matches_workspace_entry_point_twice(mode):
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=4, context=1500)
    r = LayerRun(w, mode)
    r.write()
    ref_out = r.decode(num_workers=0)           # caller workspace, planned workers
    ref = ref_out.cpu().numpy().astype(np.float64)
    pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    tol = r.tolerance(r.oracle_decode(pairs), pairs).reshape(ref.shape)
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        _fixed(r, out, r.workers)
        torch.cuda.synchronize()
        assert K().kvq_get_device_error() == 0
        check_attention(out.cpu().numpy(), ref, tol, where=f"fixed scratch call {call}")


def test_fixed_scratch_full_size_llama8b():
    w = wl.CONFIGS["llama8b"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    ref_out = r.decode(num_workers=0)
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))     # each call must write every row
        _fixed(r, out, 0)
        torch.cuda.synchronize()
        pairs = sample_pairs(w, 24, seed=5)
        got = out.cpu().numpy()
        r.check_decode(out, pairs=pairs, where="fixed scratch full size")
        assert np.allclose(got, ref_out.cpu().numpy(), rtol=1e-5, atol=1e-5)


def test_fixed_scratch_refuses_a_plan_that_does_not_fit():
    kvq = K()
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=2, context=64)
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    r.write()
    out = torch.zeros(w.B, w.Hq, w.D, device="cuda")
    r.q = wl.queries(w, "cuda")
    workers = 20000                 # partials far beyond the 16 MiB array
    _, need = kvq.kvq_decode_plan(r.ctx, 0, w.B, 64, workers)
    assert need > 16 * 1024 * 1024
    with pytest.raises(kvq.KVQError, match="WORKSPACE"):
        _fixed(r, out, workers)
    assert torch.all(out == 0)


def test_fixed_scratch_automatic_plan_shrinks_to_fit():
    """With num_workers = 0 the automatic plan is cut to what the array holds:
    here 1024 sequences x 8 KV heads at D = 256 need more than 16 MiB for the
    per-item slots alone, so the call runs on one worker (no scratch) and
    still matches the workspace entry point."""
    kvq = K()
    w = wl.Workload("wide256", Hq=16, Hkv=8, D=256, block_size=16,
                    context_lens=tuple([40] * 1024), windows=(0,), seed=97)
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    _, need = kvq.kvq_decode_plan(r.ctx, 0, w.B, 40, 0)
    r.write()
    ref_out = r.decode(num_workers=0)
    assert r.workers > 1 and need > 16 * 1024 * 1024
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        _fixed(r, out, 0)
        torch.cuda.synchronize()
        assert K().kvq_get_device_error() == 0
        assert torch.allclose(out, ref_out, rtol=1e-5, atol=1e-5)
    r.check_decode(out, pairs=sample_pairs(w, 32, seed=3), where="fixed scratch shrunk plan")
