"""Shared test plumbing: host copies of the seeded workloads for the oracle."""
import json
import os

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


# ---------------------------------------------------------------- tolerance
LOG2E = 1.4426950408889634
U32 = 2.0 ** -24


def attention_tolerance(q_row, K, V, ref_row, softmax_scale, atol=2e-3):
    """Per-output-row tolerance for an fp32 kernel against the float64 oracle.

    atol (2e-3) plus first-order fp32 forward-error terms of the kernels'
    arithmetic, each a probabilistic bound (square root of the number of
    roundings, times 4):
      * score of position i: D/16 tensor-core accumulation steps and about
        three more roundings, each at most u a_i with a_i = sum_d |q_d K_id|
        (log2 units); a score error ds_i moves the output by
        ln2 * ds_i * w_i |V_i - o|, so the term is
        4 sqrt(D/16 + 3) u ln2 sum_i w_i a_i |V_i - o|;
      * weights and values: each weight meets V with a relative error of a
        few u (exponent, scale products, the 22-bit hi + lo split: 8u), and
        the weighted sum accumulates over n/16 position tiles plus the
        split-K merge: (8 + 4 sqrt(n/16 + 2)) u sum_i w_i |V_i|;
      * normalisation: 4u |o|.
    u = 2^-24, w_i the float64 softmax weights, n the retained positions.
    For rows whose values are O(1) this is atol; it only widens for heads
    whose scores and values reach the hundreds, where an absolute 2e-3 asks
    for more than fp32 scores carry.  tests/test_tolerance_discriminates.py
    shows it still rejects a single-f16 weight, bf16 keys and f16 scores.
    q_row [D], K/V [n, D] float64 (dequantized), ref_row [D].
    """
    n, D = K.shape
    if n == 0:
        return np.full(D, atol)
    a = np.abs(K) @ np.abs(q_row) * softmax_scale * LOG2E
    s = (K @ q_row) * softmax_scale
    w = np.exp(s - s.max())
    w /= w.sum()
    spread = (w * a) @ np.abs(V - ref_row[None, :])
    mag = w @ np.abs(V)
    return atol + 4 * np.sqrt(D / 16 + 3) * U32 * np.log(2) * spread \
        + (8 + 4 * np.sqrt(n / 16 + 2)) * U32 * mag + 4 * U32 * np.abs(ref_row)


def check_attention(got, ref, tol, where="", flat=False, atol=2e-3):
    """Element-wise |got-ref| <= tol and relative L2 <= 1e-3 over the tensor;
    with flat=True every element must also be within the flat atol.  Returns
    (max |err|, relative L2) and, when KVQ_PARITY_REPORT names a file,
    appends them there with the count of elements over atol."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > tol
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    over = int((err > atol).sum())
    path = os.environ.get("KVQ_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": where, "elements": int(err.size),
                                "max_abs_err": float(err.max()) if err.size else 0.0,
                                "rel_l2": float(rel), "elements_over_2e-3": over,
                                "flat": bool(flat)}) + "\n")
    assert not bad.any(), (f"{where}: {bad.sum()} elements over tolerance; worst err "
                           f"{err.max():.3e} (tol there {tol.flat[err.argmax()]:.3e})")
    assert rel <= 1e-3, f"{where}: relative L2 {rel:.3e}"
    if flat:
        assert over == 0, f"{where}: {over} elements over the flat {atol:g}, worst {err.max():.3e}"
    return float(err.max()), float(rel)
