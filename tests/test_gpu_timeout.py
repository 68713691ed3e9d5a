"""The bounded device wait runs out, reports KVQ_ERR_TIMEOUT and leaves the
context usable.

Every barrier wait in the kernels is bounded (about 2 s) so that a copy that
never lands cannot hang the GPU.  kvq_check_bounded_wait runs that same wait
on a barrier that expects bytes no copy delivers, with a limit of about 1 ms;
no copy is issued, so nothing is in flight when it gives up.
"""
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_sets_timeout_and_context_survives():
    kvq = K()
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    kvq.kvq_check_bounded_wait(2_000_000)
    assert kvq.STATUS[kvq.kvq_get_device_error()] == "KVQ_ERR_TIMEOUT"
    # the word was cleared by the read, and the context still runs kernels
    assert kvq.kvq_get_device_error() == 0
    r = LayerRun(wl.CONFIGS["tiny"], orc.FP8_PER_TOKEN_HEAD)
    r.write()
    r.check_write()
    r.check_decode(r.decode())


def test_wait_limit_is_validated():
    kvq = K()
    for bad in (0, -5, (1 << 31) + 1):
        with pytest.raises(kvq.KVQError, match="INVALID_ARG"):
            kvq.kvq_check_bounded_wait(bad)
