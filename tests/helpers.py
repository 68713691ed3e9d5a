"""Shared test plumbing: host copies of the seeded workloads for the oracle."""
import numpy as np
import torch

from int4_quantized_paged_gb300 import workloads as wl


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def host_fill(w: wl.Workload, layer: int = 0, device="cpu"):
    """Whole-context fill inputs for one layer, as host arrays."""
    pg = wl.paging(w, device)
    pos = wl.fill_positions(w)
    T = sum(len(p) for p in pos)
    k, v = wl.kv_tokens(w, T, device, layer=layer)
    slots = wl.slot_mapping(w, pg, pos, device)
    return {
        "k": k, "v": v, "slots": slots, "paging": pg, "T": T,
        "k_bits": bits(k), "v_bits": bits(v), "slots_np": slots.cpu().numpy(),
        "block_table": pg.block_table.cpu().numpy(), "context_lens": pg.context_lens.cpu().numpy(),
    }
