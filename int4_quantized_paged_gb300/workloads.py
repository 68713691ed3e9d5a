"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws inputs and nothing else: no quantization, no attention and
no scale arithmetic live here.  The tests feed the same tensors (host copies)
to the CPU oracle and the CUDA library; ``bench.py`` uses the same recipes.

Recipe (all seeded; one torch.Generator per tensor, seeded from the config
seed and a fixed stream number, on the device the tensors are made on):

* Q, K, V base values ~ N(0, 1), drawn in fp32 and rounded to bf16.
* Per-KV-head multipliers: a fixed head list (tiny config: head 1 x16) or a
  log-uniform draw in [lo, hi] per KV head; the same multiplier scales that
  head's K and V.  Q is never scaled.
* Outlier tokens: a Bernoulli(p) draw per token position; an outlier token's K
  and V are multiplied by the factor in every head.
* Paging: physical blocks are a seeded random permutation of the pool, handed
  to the sequences in order; block-table entries past a sequence's last block
  are -1.  Slot mapping of position p of sequence b is
  block_table[b, p // bs] * bs + p % bs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

MODES = {"bf16": 0, "fp8_per_tensor": 1, "fp8_per_head": 2, "fp8_per_token_head": 3,
         "int4_per_token_head": 4}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    Hq: int
    Hkv: int
    D: int
    block_size: int
    context_lens: tuple          # one entry per sequence
    windows: tuple = (0,)        # one entry per layer, 0 = full attention
    head_mult: Optional[tuple] = None      # explicit per-KV-head multipliers
    head_mult_loguniform: Optional[tuple] = None  # (lo, hi)
    outlier_p: float = 0.0
    outlier_factor: float = 1.0
    seed: int = 1234
    write_tokens_per_seq: int = 0  # prefill-shaped write size (0: whole context)

    @property
    def B(self) -> int:
        return len(self.context_lens)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def num_layers(self) -> int:
        return len(self.windows)


def _ctx(b, L):
    return tuple([L] * b)


# The five configurations.  Sizes follow the pages' workloads; see the
# design notes for where each comes from.
CONFIGS = {
    "tiny": Workload("tiny", Hq=4, Hkv=2, D=64, block_size=16, context_lens=(37, 100),
                     head_mult=(1.0, 16.0), outlier_p=0.05, outlier_factor=4.0, seed=1235),
    "llama8b": Workload("llama8b", Hq=32, Hkv=8, D=128, block_size=16,
                        context_lens=_ctx(64, 4096), head_mult_loguniform=(0.5, 32.0),
                        outlier_p=0.01, outlier_factor=8.0, seed=1236),
    "llama70b_128k": Workload("llama70b_128k", Hq=64, Hkv=8, D=128, block_size=16,
                              context_lens=_ctx(8, 131072), head_mult_loguniform=(0.5, 32.0),
                              seed=1237),
    "gptoss20b": Workload("gptoss20b", Hq=64, Hkv=8, D=64, block_size=16,
                          context_lens=_ctx(16, 32768), windows=tuple([128, 0] * 12), seed=1238),
    "gemma_d256": Workload("gemma_d256", Hq=16, Hkv=8, D=256, block_size=16,
                           context_lens=_ctx(32, 16384), windows=(512, 0),
                           head_mult_loguniform=(0.5, 32.0), outlier_p=0.01, outlier_factor=8.0,
                           seed=1239, write_tokens_per_seq=8192),
}


def scaled(w: Workload, batch: Optional[int] = None, context: Optional[int] = None) -> Workload:
    """Same recipe at a smaller batch / context (parity cases the oracle finishes)."""
    b = w.B if batch is None else batch
    L = w.context_lens[0] if context is None else context
    cl = w.context_lens[:b] if context is None else _ctx(b, L)
    wt = min(w.write_tokens_per_seq, L) if w.write_tokens_per_seq else 0
    return dataclasses.replace(w, context_lens=tuple(cl), write_tokens_per_seq=wt)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + stream)
    return g


def head_multipliers(w: Workload) -> torch.Tensor:
    """Per-KV-head multipliers (fp32, CPU), same for K and V."""
    if w.head_mult is not None:
        return torch.tensor(w.head_mult, dtype=torch.float32)
    if w.head_mult_loguniform is not None:
        lo, hi = w.head_mult_loguniform
        u = torch.rand(w.Hkv, generator=_gen("cpu", w.seed, 1), dtype=torch.float64)
        return torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).float()
    return torch.ones(w.Hkv, dtype=torch.float32)


def outlier_factors(w: Workload, n_tokens: int, stream: int, device) -> torch.Tensor:
    """Per-token factor (fp32): outlier_factor with probability outlier_p, else 1."""
    if w.outlier_p <= 0.0:
        return torch.ones(n_tokens, dtype=torch.float32, device=device)
    u = torch.rand(n_tokens, generator=_gen(device, w.seed, stream), device=device)
    one = torch.ones((), device=device)
    return torch.where(u < w.outlier_p, one * w.outlier_factor, one)


def kv_tokens(w: Workload, n_tokens: int, device, layer: int = 0, stream_base: int = 10):
    """New K and V vectors [n_tokens, Hkv, D] bf16 for one layer."""
    mult = head_multipliers(w).to(device)
    s = stream_base + 8 * layer
    fac = outlier_factors(w, n_tokens, s + 2, device)
    out = []
    for j in range(2):
        x = torch.randn(n_tokens, w.Hkv, w.D, generator=_gen(device, w.seed, s + j),
                        device=device, dtype=torch.float32)
        x = x * mult[None, :, None] * fac[:, None, None]
        out.append(x.to(torch.bfloat16))
    return out[0], out[1]


def queries(w: Workload, device, layer: int = 0) -> torch.Tensor:
    """Decode queries [B, Hq, D] bf16 ~ N(0, 1)."""
    g = _gen(device, w.seed, 500 + layer)
    return torch.randn(w.B, w.Hq, w.D, generator=g, device=device).to(torch.bfloat16)


def calibration_sample(w: Workload, device, n_tokens: int = 512, layer: int = 0):
    """A separate seeded draw of n_tokens K/V tokens from the same recipe
    (used to derive static per-head scales)."""
    return kv_tokens(w, n_tokens, device, layer=layer, stream_base=900)


@dataclasses.dataclass
class Paging:
    block_table: torch.Tensor   # int32 [B, max_blocks], -1 past the end
    context_lens: torch.Tensor  # int32 [B]
    num_blocks: int
    max_blocks: int


def paging(w: Workload, device, spare_blocks: int = 0) -> Paging:
    bs = w.block_size
    nb = [(L + bs - 1) // bs for L in w.context_lens]
    total = sum(nb) + spare_blocks
    maxb = max(max(nb), 1)
    perm = torch.randperm(total, generator=_gen("cpu", w.seed, 2)).to(torch.int32)
    bt = torch.full((w.B, maxb), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nb):
        bt[b, :n] = perm[off:off + n]
        off += n
    cl = torch.tensor(w.context_lens, dtype=torch.int32)
    return Paging(bt.to(device), cl.to(device), total, maxb)


def ring_paging(w: Workload, window: int, device) -> Paging:
    """Paging of a window layer that reuses freed blocks: sequence b owns a
    ring of R = ceil(W / bs) + 1 physical blocks and logical block j maps to
    ring slot j mod R.  When position p is written, the block it overwrites
    held positions below p + 1 - W, outside the window, so the retained
    positions [L - W, L) always sit in distinct live blocks."""
    bs = w.block_size
    R = (window + bs - 1) // bs + 1
    nb = [(L + bs - 1) // bs for L in w.context_lens]
    maxb = max(max(nb), 1)
    perm = torch.randperm(w.B * R, generator=_gen("cpu", w.seed, 3)).to(torch.int32)
    bt = torch.full((w.B, maxb), -1, dtype=torch.int32)
    for b, n in enumerate(nb):
        ring = perm[b * R:(b + 1) * R]
        bt[b, :n] = ring[torch.arange(n) % R]
    cl = torch.tensor(w.context_lens, dtype=torch.int32)
    return Paging(bt.to(device), cl.to(device), w.B * R, maxb)


def slot_mapping(w: Workload, pg: Paging, positions: Sequence[range], device) -> torch.Tensor:
    """int64 slots for the given positions of each sequence, sequence-major."""
    bt = pg.block_table.cpu()
    bs = w.block_size
    parts = []
    for b, pos in enumerate(positions):
        p = torch.tensor(list(pos), dtype=torch.int64) if not isinstance(pos, torch.Tensor) else pos
        if p.numel() == 0:
            continue
        blk = bt[b, p // bs].to(torch.int64)
        parts.append(blk * bs + p % bs)
    if not parts:
        return torch.zeros(0, dtype=torch.int64, device=device)
    return torch.cat(parts).to(device)


def fill_positions(w: Workload):
    """Positions written by a whole-context fill: [0, L_b) for each sequence."""
    return [torch.arange(L, dtype=torch.int64) for L in w.context_lens]
