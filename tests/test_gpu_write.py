"""GPU cache write against the oracle: codes and scales bit-exact.

Cases span the five workloads (scaled down where the oracle must finish in
seconds, and at full size for the prefill-shaped fills the benchmark times),
every scale mode, ragged tails and skipped slots.
"""
import numpy as np
import pytest
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.gpu_harness import K, LayerRun
from tests.helpers import bits

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": wl.CONFIGS["tiny"],
    "llama8b": wl.scaled(wl.CONFIGS["llama8b"], batch=3, context=1000),
    "llama70b": wl.scaled(wl.CONFIGS["llama70b_128k"], batch=2, context=2500),
    "gptoss": wl.scaled(wl.CONFIGS["gptoss20b"], batch=3, context=700),
    "gemma": wl.scaled(wl.CONFIGS["gemma_d256"], batch=2, context=1200),
}
MODES = [orc.BF16, orc.FP8_PER_TENSOR, orc.FP8_PER_HEAD, orc.FP8_PER_TOKEN_HEAD,
         orc.INT4_PER_TOKEN_HEAD]


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode", MODES)
def test_write_bit_exact_small(name, mode):
    r = LayerRun(SMALL[name], mode)
    r.write()
    r.check_write()


# Writes of fewer chunks than SMs take the direct kernel (registers hold the
# rows), larger ones the staged kernel (rows streamed through shared memory);
# SMALL covers both (tiny and gptoss direct, the others staged).  These add
# the direct path at D = 128 and 256 in every mode.
DIRECT = {
    "llama8b_b1": wl.scaled(wl.CONFIGS["llama8b"], batch=1, context=200),
    "gemma_b1": wl.scaled(wl.CONFIGS["gemma_d256"], batch=1, context=300),
}


@pytest.mark.parametrize("name", list(DIRECT))
@pytest.mark.parametrize("mode", MODES)
def test_write_bit_exact_direct_path(name, mode):
    r = LayerRun(DIRECT[name], mode)
    r.write()
    r.check_write()


@pytest.mark.parametrize("mode", [orc.FP8_PER_TENSOR, orc.FP8_PER_HEAD, orc.FP8_PER_TOKEN_HEAD])
def test_write_bit_exact_llama8b_full_fill(mode):
    r = LayerRun(wl.CONFIGS["llama8b"], mode)
    r.write()
    r.check_write()


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD])
def test_write_bit_exact_gemma_prefill_chunk(mode):
    # Prefill-shaped write: 8192 new tokens per sequence at positions [8192, 16384)
    # of 32 sequences, on top of a fill of [0, 8192).
    w = wl.CONFIGS["gemma_d256"]
    r = LayerRun(w, mode, layer=1)
    first = [torch.arange(0, 8192) for _ in range(w.B)]
    second = [torch.arange(8192, 16384) for _ in range(w.B)]
    r.write(first)
    r_host_first = r.host
    # second chunk: new seeded tokens through both paths into the same caches
    kvq = K()
    T = 8192 * w.B
    k, v = wl.kv_tokens(w, T, "cuda", layer=1, stream_base=300)
    slots = wl.slot_mapping(w, r.pg, second, "cuda")
    kvq.kvq_cache_write(r.ctx, 1, k, v, slots, r.kc, r.vc, r.ks, r.vs)
    torch.cuda.synchronize()
    kc, vc, ks, vs = r_host_first
    orc.cache_write(mode, bits(k), bits(v), slots.cpu().numpy(), kc, vc, ks, vs)
    r.check_write()


def test_negative_slots_skip_and_canaries_survive():
    w = SMALL["llama8b"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    for t in (r.kc, r.vc):
        t.fill_(0xA5)
    for t in (r.ks, r.vs):
        t.fill_(-3.0)
    kvq = K()
    pos = wl.fill_positions(w)
    T = sum(len(p) for p in pos)
    k, v = wl.kv_tokens(w, T, "cuda")
    slots = wl.slot_mapping(w, r.pg, pos, "cuda")
    skip = torch.arange(T, device="cuda") % 5 == 2
    slots_m = torch.where(skip, torch.full_like(slots, -1), slots)
    kvq.kvq_cache_write(r.ctx, 0, k, v, slots_m, r.kc, r.vc, r.ks, r.vs)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    kc, vc, ks, vs = orc.alloc_cache(orc.FP8_PER_TOKEN_HEAD, r.pg.num_blocks, w.Hkv, 16, w.D)
    kc[:] = 0xA5; vc[:] = 0xA5; ks[:] = -3.0; vs[:] = -3.0
    orc.cache_write(orc.FP8_PER_TOKEN_HEAD, bits(k), bits(v), slots_m.cpu().numpy(), kc, vc, ks, vs)
    r.host = (kc, vc, ks, vs)
    r.check_write()


def test_slot_past_the_cache_is_reported_not_written():
    w = SMALL["tiny"]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    kvq = K()
    k, v = wl.kv_tokens(w, 4, "cuda")
    cap = r.pg.num_blocks * w.block_size
    slots = torch.tensor([0, cap, cap + 100, 5], dtype=torch.int64, device="cuda")
    kvq.kvq_cache_write(r.ctx, 0, k, v, slots, r.kc, r.vc, r.ks, r.vs)
    assert kvq.kvq_get_device_error() == kvq.STATUS.index("KVQ_ERR_BAD_INDEX")
    assert kvq.kvq_get_device_error() == 0          # the word was cleared
    kc, vc, ks, vs = orc.alloc_cache(orc.FP8_PER_TOKEN_HEAD, r.pg.num_blocks, w.Hkv, 16, w.D)
    good = np.array([0, -1, -1, 5])
    orc.cache_write(orc.FP8_PER_TOKEN_HEAD, bits(k), bits(v), good, kc, vc, ks, vs)
    r.host = (kc, vc, ks, vs)
    r.check_write()


def test_slot_past_the_cache_staged_path():
    w = SMALL["llama8b"]
    r = LayerRun(w, orc.INT4_PER_TOKEN_HEAD)
    kvq = K()
    pos = wl.fill_positions(w)
    T = sum(len(p) for p in pos)
    k, v = wl.kv_tokens(w, T, "cuda")
    slots = wl.slot_mapping(w, r.pg, pos, "cuda")
    cap = r.pg.num_blocks * w.block_size
    bad = torch.tensor([7, 1500, T - 1], device="cuda")
    slots[bad] = torch.tensor([cap, cap + 5, 1 << 40], dtype=torch.int64, device="cuda")
    kvq.kvq_cache_write(r.ctx, 0, k, v, slots, r.kc, r.vc, r.ks, r.vs)
    assert kvq.kvq_get_device_error() == kvq.STATUS.index("KVQ_ERR_BAD_INDEX")
    good = slots.cpu().numpy().copy()
    good[bad.cpu().numpy()] = -1
    kc, vc, ks, vs = orc.alloc_cache(orc.INT4_PER_TOKEN_HEAD, r.pg.num_blocks, w.Hkv, 16, w.D)
    orc.cache_write(orc.INT4_PER_TOKEN_HEAD, bits(k), bits(v), good, kc, vc, ks, vs)
    r.host = (kc, vc, ks, vs)
    r.check_write()


@pytest.mark.parametrize("name", ["llama8b", "tiny"])
def test_strided_token_rows(name):
    # K and V as column slices of one [T, 3, Hkv*D] projection output
    # (llama8b: staged path; tiny: direct path).
    w = SMALL[name]
    r = LayerRun(w, orc.FP8_PER_TOKEN_HEAD)
    kvq = K()
    pos = wl.fill_positions(w)
    T = sum(len(p) for p in pos)
    k, v = wl.kv_tokens(w, T, "cuda")
    qkv = torch.zeros(T, 3, w.Hkv * w.D, dtype=torch.bfloat16, device="cuda")
    qkv[:, 1] = k.reshape(T, -1)
    qkv[:, 2] = v.reshape(T, -1)
    slots = wl.slot_mapping(w, r.pg, pos, "cuda")
    kvq.kvq_cache_write(r.ctx, 0, qkv[:, 1], qkv[:, 2], slots, r.kc, r.vc, r.ks, r.vs,
                        kv_token_stride=3 * w.Hkv * w.D)
    torch.cuda.synchronize()
    kc, vc, ks, vs = orc.alloc_cache(orc.FP8_PER_TOKEN_HEAD, r.pg.num_blocks, w.Hkv, 16, w.D)
    orc.cache_write(orc.FP8_PER_TOKEN_HEAD, bits(k), bits(v), slots.cpu().numpy(), kc, vc, ks, vs)
    r.host = (kc, vc, ks, vs)
    r.check_write()


def test_e4m3_encoder_all_fp32_bit_patterns():
    """The device encoder against the oracle's software encoder on all 2^32
    fp32 patterns (NaN inputs: only the NaN-ness of the code is compared)."""
    kvq = K()
    chunk = 1 << 28
    inp = torch.empty(chunk, dtype=torch.int32, device="cuda")
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    base = torch.arange(chunk, dtype=torch.int64, device="cuda")
    ora = orc.lib()
    for c in range(1 << 4):
        x = (base + c * chunk)
        inp.copy_((x - (1 << 32) * (x >= (1 << 31))).to(torch.int32))
        kvq.kvq_e4m3_encode(inp.view(torch.float32), out)
        got = out.cpu().numpy()
        f = inp.cpu().numpy().view(np.float32)
        ref = np.empty(chunk, dtype=np.uint8)
        ora.orc_e4m3_encode_array(f.ctypes.data, ref.ctypes.data, chunk)
        nan = np.isnan(f)
        assert np.array_equal(got[~nan], ref[~nan]), f"chunk {c}"
        assert np.all((got[nan] & 0x7F) == 0x7F), f"chunk {c} NaN"


@pytest.mark.parametrize("mode", [orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD])
def test_dynamic_scale_every_bf16_amax(mode):
    # One vector per positive finite bf16 amax (all 32639 of them, subnormal to
    # the largest), with random bf16 elements below it: every dynamic scale
    # the write can compute, both the reciprocal paths and the division
    # fallback for tiny amax, bit-exact against the oracle.
    w = wl.Workload("edges", Hq=8, Hkv=8, D=128, block_size=16, context_lens=(1360, 1360, 1360))
    r = LayerRun(w, mode)
    g = torch.Generator().manual_seed(9)
    T = sum(w.context_lens)
    amax_bits = torch.arange(1, 0x7F80, dtype=torch.int64)                 # every bf16 > 0
    amax_bits = torch.cat([amax_bits, amax_bits[:T * w.Hkv - amax_bits.numel()]])
    k_bits = amax_bits[torch.randperm(amax_bits.numel(), generator=g)]
    v_bits = amax_bits[torch.randperm(amax_bits.numel(), generator=g)]

    def vectors(ab):
        amax = (ab.to(torch.int32) << 16).view(torch.float32).reshape(T, w.Hkv, 1)
        frac = torch.rand(T, w.Hkv, w.D, generator=g) * 2 - 1
        x = (frac * amax).to(torch.bfloat16)
        x[..., 5] = (-amax[..., 0]).to(torch.bfloat16)      # the amax, negative, mid-vector
        return x.cuda()
    k, v = vectors(k_bits), vectors(v_bits)
    pos = wl.fill_positions(w)
    slots = wl.slot_mapping(w, r.pg, pos, "cuda")
    kvq = K()
    kvq.kvq_cache_write(r.ctx, 0, k, v, slots, r.kc, r.vc, r.ks, r.vs)
    torch.cuda.synchronize()
    kc, vc, ks, vs = orc.alloc_cache(mode, r.pg.num_blocks, w.Hkv, 16, w.D)
    orc.cache_write(mode, bits(k), bits(v), slots.cpu().numpy(), kc, vc, ks, vs)
    r.host = (kc, vc, ks, vs)
    r.check_write()


@pytest.mark.parametrize("scale", [2.0 ** -90, 2.0 ** -70, 3.1e-9, 0.0123, 7.5, 2.0 ** 40, 2.0 ** 110])
def test_static_scale_extremes(scale):
    w = SMALL["llama8b"]
    r = LayerRun(w, orc.FP8_PER_TENSOR, per_tensor_scale=scale)
    r.write()
    r.check_write()
