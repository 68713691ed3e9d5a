"""Runs one layer of a workload through the C ABI on the GPU and through the
CPU oracle on host copies of the same seeded inputs, and compares them.

The oracle never sees anything the GPU computed: it gets the generator's
inputs (host copies) and writes its own cache from them.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

from int4_quantized_paged_gb300 import workloads as wl
from oracle import oracle as orc
from tests.helpers import attention_tolerance, bf16_to_f64, bits, check_attention


# Workload recipes on which the decode meets the flat max-abs 2e-3 in every
# mode (measured at full size over every output row).  The Llama-8B-like
# recipe is not among them: its x32 heads with x8 outlier positions reach
# outputs of several hundred, where some rows need scores more exact than
# fp32 holds (tests/test_tolerance_discriminates.py shows that even scores
# rounded once to fp32 miss 2e-3 there); those rows are held to the per-row
# bound.
FLAT_WORKLOADS = {"tiny", "llama70b_128k", "gptoss20b", "gemma_d256"}


def K():
    from int4_quantized_paged_gb300 import kvq
    return kvq


@dataclasses.dataclass
class LayerRun:
    w: wl.Workload
    mode: int
    layer: int = 0
    per_tensor_scale: float = 1.0       # control value for FP8_PER_TENSOR
    device: str = "cuda"

    def __post_init__(self):
        kvq = K()
        w = self.w
        modes = [self.mode] * w.num_layers
        self.window = w.windows[self.layer]
        self.pg = wl.paging(w, self.device)
        self.ctx = kvq.kvq_create(w.num_layers, w.Hq, w.Hkv, w.D, w.block_size,
                                  self.pg.num_blocks, modes, list(w.windows))
        self.kc, self.vc, self.ks, self.vs = kvq.alloc_layer_cache(self.ctx, self.layer,
                                                                  self.device)
        self.k_scale = self.v_scale = None
        self.o_k_scale = self.o_v_scale = None
        self.host = None

    # ------------------------------------------------------------ scales
    def static_scales(self):
        """Per-tensor: the control constant on both sides.  Per-head: each side
        calibrates from the same 512-token sample; the results must agree."""
        kvq = K()
        w = self.w
        if self.mode == orc.FP8_PER_TENSOR:
            one = np.array([self.per_tensor_scale], dtype=np.float32)
            self.o_k_scale = self.o_v_scale = one
            self.k_scale = torch.tensor(one, device=self.device)
            self.v_scale = self.k_scale.clone()
        elif self.mode == orc.FP8_PER_HEAD:
            ck, cv = wl.calibration_sample(w, self.device, layer=self.layer)
            self.k_scale = torch.empty(w.Hkv, dtype=torch.float32, device=self.device)
            self.v_scale = torch.empty_like(self.k_scale)
            kvq.kvq_calibrate_per_head(self.ctx, ck, self.k_scale)
            kvq.kvq_calibrate_per_head(self.ctx, cv, self.v_scale)
            self.o_k_scale = orc.calibrate_per_head(bits(ck))
            self.o_v_scale = orc.calibrate_per_head(bits(cv))
            assert np.array_equal(self.k_scale.cpu().numpy(), self.o_k_scale)
            assert np.array_equal(self.v_scale.cpu().numpy(), self.o_v_scale)

    # ------------------------------------------------------------ write
    def write(self, positions: Optional[Sequence] = None):
        """GPU write through kvq_cache_write and oracle write of the same tokens."""
        kvq = K()
        w = self.w
        self.static_scales()
        pos = wl.fill_positions(w) if positions is None else positions
        T = sum(len(p) for p in pos)
        k, v = wl.kv_tokens(w, T, self.device, layer=self.layer)
        slots = wl.slot_mapping(w, self.pg, pos, self.device)
        kvq.kvq_cache_write(self.ctx, self.layer, k, v, slots, self.kc, self.vc, self.ks, self.vs,
                            self.k_scale, self.v_scale)
        torch.cuda.synchronize()
        assert kvq.kvq_get_device_error() == 0
        kc, vc, ks, vs = orc.alloc_cache(self.mode, self.pg.num_blocks, w.Hkv, w.block_size, w.D)
        orc.cache_write(self.mode, bits(k), bits(v), slots.cpu().numpy(), kc, vc, ks, vs,
                        k_scale=self.o_k_scale, v_scale=self.o_v_scale, block_size=w.block_size)
        self.host = (kc, vc, ks, vs)
        return T

    def check_write(self):
        kc, vc, ks, vs = self.host
        assert np.array_equal(self.kc.cpu().numpy(), kc), "K codes differ from the oracle"
        assert np.array_equal(self.vc.cpu().numpy(), vc), "V codes differ from the oracle"
        if ks is not None:
            gk, gv = self.ks.cpu().numpy(), self.vs.cpu().numpy()
            assert np.array_equal(gk.view(np.uint32), ks.view(np.uint32)), "K scales differ"
            assert np.array_equal(gv.view(np.uint32), vs.view(np.uint32)), "V scales differ"

    # ------------------------------------------------------------ decode
    def decode(self, num_workers: int = 0, context_lens=None, q=None):
        """GPU decode; the workspace is filled with NaN first so that a partial
        that is read without having been written shows up."""
        kvq = K()
        w = self.w
        self.q = wl.queries(w, self.device, layer=self.layer) if q is None else q
        cl = self.pg.context_lens if context_lens is None else context_lens
        self.cl = cl
        max_ctx = int(cl.max().item()) if cl.numel() else 0
        workers, ws_bytes = kvq.kvq_decode_plan(self.ctx, self.layer, w.B, max_ctx, num_workers)
        ws = torch.full((max(ws_bytes, 16) // 4,), float("nan"), dtype=torch.float32,
                        device=self.device)
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device=self.device)
        kvq.kvq_decode_attention(self.ctx, self.layer, self.q, self.kc, self.vc,
                                 self.pg.block_table, cl, out, max_context=max_ctx,
                                 k_scale=self.k_scale, v_scale=self.v_scale,
                                 k_cache_scale=self.ks, v_cache_scale=self.vs,
                                 num_workers=workers, workspace=ws)
        torch.cuda.synchronize()
        assert kvq.kvq_get_device_error() == 0
        self.workers = workers
        return out

    def oracle_decode(self, pairs=None):
        kc, vc, ks, vs = self.host
        return orc.decode(self.mode, bits(self.q), kc, vc, self.pg.block_table.cpu().numpy(),
                          self.cl.cpu().numpy(), k_scale=self.o_k_scale, v_scale=self.o_v_scale,
                          k_cache_scale=ks, v_cache_scale=vs, window=self.window,
                          block_size=self.w.block_size, pairs=pairs)

    def tolerance(self, ref, pairs):
        """Row tolerances for the given (b, hq) pairs; ref is [len(pairs), D]."""
        kc, vc, ks, vs = self.host
        w = self.w
        bt = self.pg.block_table.cpu().numpy()
        cl = self.cl.cpu().numpy()
        qd = bf16_to_f64(bits(self.q))
        tol = np.zeros_like(ref)
        cache = {}
        for i, (b, hq) in enumerate(pairs):
            g = hq // w.G
            if (b, g) not in cache:
                L = int(cl[b])
                lo = max(0, L - self.window) if self.window > 0 else 0
                p = np.arange(lo, L)
                blk, off = bt[b, p // w.block_size], p % w.block_size
                Kh = _rows(self.mode, kc, ks, self.o_k_scale, blk, g, off)
                Vh = _rows(self.mode, vc, vs, self.o_v_scale, blk, g, off)
                cache = {(b, g): (Kh, Vh)}
            Kh, Vh = cache[(b, g)]
            tol[i] = attention_tolerance(qd[b, hq], Kh, Vh, ref[i], 1.0 / np.sqrt(w.D))
        return tol

    def check_decode(self, out, pairs=None, where="", flat=None):
        """Against the oracle: the per-row bound everywhere, and the flat
        2e-3 too when `flat` (default: the workload is one measured to meet
        it, see FLAT_WORKLOADS)."""
        w = self.w
        if pairs is None:
            pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
        ref = self.oracle_decode(pairs)
        got = out.cpu().numpy()[[p[0] for p in pairs], [p[1] for p in pairs]]
        tol = self.tolerance(ref, pairs)
        if flat is None:
            flat = w.name in FLAT_WORKLOADS
        return check_attention(got, ref, tol, where or f"{w.name} mode {self.mode}", flat=flat)


def _rows(mode, codes, slot_scales, static, blk, g, off):
    """Dequantized rows (float64 [n, D]) of KV head g at (blk[i], off[i])."""
    c = codes[blk, g, off]                              # [n, row]
    if c.shape[0] == 0:
        return np.zeros((0, c.shape[1] * (2 if mode == orc.INT4_PER_TOKEN_HEAD else 1)
                         // (2 if mode == orc.BF16 else 1)))
    s = None if slot_scales is None else slot_scales[blk, g, off]
    if mode in (orc.FP8_PER_TOKEN_HEAD, orc.INT4_PER_TOKEN_HEAD):
        return orc.dequantize(mode, c[:, None, None, :], s[:, None, None])[:, 0, 0, :]
    if mode == orc.FP8_PER_HEAD:
        return orc.dequantize(orc.FP8_PER_TENSOR, c[:, None, None, :], None,
                              np.asarray([static[g]]))[:, 0, 0, :]
    return orc.dequantize(mode, c[:, None, None, :], None, static)[:, 0, 0, :]


def sample_pairs(w: wl.Workload, n: int, seed: int = 0):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, w.B, size=n)
    h = rng.integers(0, w.Hq, size=n)
    pairs = sorted(set(zip(b.tolist(), h.tolist())))
    return pairs
