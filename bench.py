"""Benchmark of the quantized paged KV cache hot path on one GB300.

One step = one decode step of the Llama-3-8B-like layer (Hq=32, Hkv=8, D=128,
block 16, batch 64 x context 4096, dynamic per-token-head FP8 by default):
kvq_cache_write of the current token of every sequence, then
kvq_decode_attention over the 4096 cached positions.  Throughput is
algorithmic bytes (what the method must move: codes, scales, q, out, block
table, new K/V and slots) per second.  The same run also times a
prefill-shaped cache write of the whole 262,144-token context (cache-write
GB/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode fp8_per_token_head]
    python bench.py --impl reference     # the CPU oracle on a bounded sample

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
work shards by sequence with no exchange); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
METRIC = ("FP8-KV decode attention GB/s and KV-tokens/s (% of HBM roofline); "
          "cache-write GB/s")
WORKLOAD = "llama8b"


# ------------------------------------------------------------------ ranks
def rank_env():
    r = int(os.environ.get("RANK", "0"))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", str(r)))
    return r, ws, lr


def init_dist(backend: str):
    import torch.distributed as dist
    _, ws, _ = rank_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return dist if ws > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ bytes
def elem_bytes(mode: int) -> float:
    return {0: 2.0, 4: 0.5}.get(mode, 1.0)


def decode_bytes(w, mode: int, window: int = 0) -> float:
    """Algorithmic bytes of one decode launch: retained K/V codes and dynamic
    scales, q (bf16), out (fp32) and the block-table entries read."""
    dyn = mode in (3, 4)
    total = 0.0
    for L in w.context_lens:
        kept = min(L, window) if window > 0 else L
        total += kept * w.Hkv * (2 * w.D * elem_bytes(mode) + (8 if dyn else 0))
        total += 4 * ((L + w.block_size - 1) // w.block_size)
    total += w.B * w.Hq * w.D * (2 + 4)
    return total


def write_bytes(w, mode: int, T: int) -> float:
    """Algorithmic bytes of writing T tokens: bf16 K/V in, codes (+ scales) out,
    int64 slot."""
    dyn = mode in (3, 4)
    return T * (w.Hkv * (4 * w.D + 2 * w.D * elem_bytes(mode) + (8 if dyn else 0)) + 8)


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        v = d.get("hbm_gbs") or d.get("hbm_GBps")
        if v:
            return float(v), "measured"
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kernel_file: str, summary: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (its sha256 is recorded in the summary)."""
    try:
        src = open(os.path.join(ROOT, "int4_quantized_paged_gb300", "csrc", kernel_file), "rb").read()
        text = open(os.path.join(ROOT, "profiles", summary)).read()
    except OSError:
        return None
    m = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != hashlib.sha256(src).hexdigest():
        return None
    return float(t.group(1))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = [l.split(",") for l in open(self.file.name).read().strip().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch
    from int4_quantized_paged_gb300 import kvq
    from int4_quantized_paged_gb300 import workloads as wl

    rank, world, local = rank_env()
    torch.cuda.set_device(local)
    dist = init_dist("nccl")
    dev = f"cuda:{local}"
    mode = kvq.MODE_NAMES[args.mode]
    base = wl.CONFIGS[WORKLOAD]
    w = wl.Workload(**{**base.__dict__, "seed": base.seed + 1000 * rank})
    L = w.context_lens[0]
    pg = wl.paging(w, dev)
    ctx = kvq.kvq_create(1, w.Hq, w.Hkv, w.D, w.block_size, pg.num_blocks, [mode])
    kc, vc, ks, vs = kvq.alloc_layer_cache(ctx, 0, dev)
    k_scale = v_scale = None
    if mode == kvq.FP8_PER_TENSOR:
        k_scale = torch.ones(1, device=dev)
        v_scale = torch.ones(1, device=dev)
    elif mode == kvq.FP8_PER_HEAD:
        ck, cv = wl.calibration_sample(w, dev)
        k_scale = torch.empty(w.Hkv, device=dev)
        v_scale = torch.empty(w.Hkv, device=dev)
        kvq.kvq_calibrate_per_head(ctx, ck, k_scale)
        kvq.kvq_calibrate_per_head(ctx, cv, v_scale)

    # whole-context fill (also the prefill-shaped write measurement)
    pos = wl.fill_positions(w)
    T_fill = sum(len(p) for p in pos)
    k_all, v_all = wl.kv_tokens(w, T_fill, dev)
    slots_all = wl.slot_mapping(w, pg, pos, dev)
    stream = torch.cuda.current_stream()

    def fill():
        kvq.kvq_cache_write(ctx, 0, k_all, v_all, slots_all, kc, vc, ks, vs, k_scale, v_scale)

    for _ in range(3):
        fill()
    torch.cuda.synchronize()
    fill_ms = []
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fill()
        e1.record(stream)
        e1.synchronize()
        fill_ms.append(e0.elapsed_time(e1))
    fill_ms_med = statistics.median(fill_ms)
    wb_fill = write_bytes(w, mode, T_fill)

    # the decode step: the current token (position L-1) of each sequence
    last = [torch.tensor([L - 1]) for _ in range(w.B)]
    idx = torch.tensor([sum(w.context_lens[:b]) + L - 1 for b in range(w.B)], device=dev)
    k_new, v_new = k_all[idx].contiguous(), v_all[idx].contiguous()
    slots_new = wl.slot_mapping(w, pg, last, dev)
    del k_all, v_all, slots_all
    q = wl.queries(w, dev)
    out = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32, device=dev)
    workers, ws_bytes = kvq.kvq_decode_plan(ctx, 0, w.B, L, args.workers)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    launches_per_step = 3          # write, decode, merge

    def step(qt=q, kn=k_new, vn=v_new, sl=slots_new, bt=pg.block_table, cl=pg.context_lens,
             o=out):
        kvq.kvq_cache_write(ctx, 0, kn, vn, sl, kc, vc, ks, vs, k_scale, v_scale)
        kvq.kvq_decode_attention(ctx, 0, qt, kc, vc, bt, cl, o, max_context=L, k_scale=k_scale,
                                 v_scale=v_scale, k_cache_scale=ks, v_cache_scale=vs,
                                 num_workers=workers, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kvq.kvq_get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(dist, local)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(n):
        ev[i][0].record(stream)
        kvq.kvq_cache_write(ctx, 0, k_new, v_new, slots_new, kc, vc, ks, vs, k_scale, v_scale)
        ev[i][1].record(stream)
        kvq.kvq_decode_attention(ctx, 0, q, kc, vc, pg.block_table, pg.context_lens, out,
                                 max_context=L, k_scale=k_scale, v_scale=v_scale,
                                 k_cache_scale=ks, v_cache_scale=vs, num_workers=workers,
                                 workspace=ws)
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, local)
    total_ms = t0.elapsed_time(t1)
    clocks = sampler.stop()
    write_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    if kvq.kvq_get_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")

    # end to end through the C ABI with host buffers
    pin = lambda t: t.cpu().pin_memory()
    h_in = [pin(x) for x in (q, k_new, v_new, slots_new, pg.block_table, pg.context_lens)]
    d_in = [torch.empty_like(x, device=dev) for x in h_in]
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = h_out.numel() * h_out.element_size()
    for _ in range(args.warmup):
        for d, h in zip(d_in, h_in):
            d.copy_(h, non_blocking=True)
        step(*d_in, o=out)
        h_out.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    barrier(dist, local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        for d, h in zip(d_in, h_in):
            d.copy_(h, non_blocking=True)
        step(*d_in, o=out)
        h_out.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n

    # ---- numbers
    ms_step = max_over_ranks(dist, total_ms / n)
    e2e_ms = max_over_ranks(dist, e2e_ms)
    dbytes = decode_bytes(w, mode)
    wbytes = write_bytes(w, mode, w.B)
    step_bytes = dbytes + wbytes
    all_bytes = sum_over_ranks(dist, step_bytes)
    kv_tokens = sum_over_ranks(dist, float(sum(w.context_lens)))
    dec_avg = statistics.mean(dec_ms)
    peak, peak_src = peak_hbm()
    dec_gbs = dbytes / (dec_avg * 1e-3) / 1e9
    fill_gbs = wb_fill / (fill_ms_med * 1e-3) / 1e9
    traffic = profiled_traffic("decode.cu", f"decode_{WORKLOAD}_{args.mode}.md")
    res = {
        "metric": METRIC,
        "value": round(all_bytes / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": n,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if mode in (1, 2, 3) else ("int4" if mode == 4 else "bf16"),
        "data": "synthetic (seeded N(0,1) x per-head log-uniform [0.5,32], 1% tokens x8)",
        "config": {"workload": "llama8b-like decode step: Hq=32 Hkv=8 D=128 block 16, "
                               "batch 64 x context 4096, 1 query/seq",
                   "mode": args.mode, "num_workers": workers,
                   "l2": "inputs larger than L2: %.0f MB of cache read per step vs 129 MB L2"
                         % (dbytes / 1e6),
                   "parallelism": f"replicas x{world} (no exchange)"},
        "kv_tokens_per_s": round(kv_tokens / (ms_step * 1e-3), 1),
        "decode": {"gbs": round(dec_gbs, 2), "ms": round(dec_avg, 5),
                   "bytes_per_launch": dbytes, "frac_of_peak": round(dec_gbs / peak, 4)},
        "write_step": {"gbs": round(wbytes / (statistics.mean(write_ms) * 1e-3) / 1e9, 2),
                       "ms": round(statistics.mean(write_ms), 5), "tokens": w.B},
        "write_fill": {"gbs": round(fill_gbs, 2), "ms": round(fill_ms_med, 4), "tokens": T_fill,
                       "bytes": wb_fill, "frac_of_peak": round(fill_gbs / peak, 4)},
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "kernel": "decode_kernel (+ log-sum-exp merge)",
                     "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": round(all_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": launches_per_step * n,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args, mode)
    if dist is not None:
        dist.destroy_process_group()
    return res if rank == 0 else None


# ------------------------------------------------------------------ oracle arm
def oracle_step_setup(mode: int, n_seq: int):
    """Bounded sample of the same workload for the CPU oracle: n_seq of the 64
    sequences, their whole 4096-token cache written by the oracle (untimed)."""
    import numpy as np
    import torch
    from int4_quantized_paged_gb300 import workloads as wl
    from oracle import oracle as orc

    base = wl.CONFIGS[WORKLOAD]
    w = wl.Workload(**{**base.__dict__, "context_lens": base.context_lens[:n_seq]})
    pg = wl.paging(w, "cpu")
    pos = wl.fill_positions(w)
    T = sum(len(p) for p in pos)
    k, v = wl.kv_tokens(w, T, "cpu")
    slots = wl.slot_mapping(w, pg, pos, "cpu").numpy()
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    kb, vb = u16(k), u16(v)
    kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, w.Hkv, w.block_size, w.D)
    sk = sv = None
    if mode == 1:
        sk = sv = np.ones(1, dtype=np.float32)
    elif mode == 2:
        ck, cv = wl.calibration_sample(base, "cpu")
        sk, sv = orc.calibrate_per_head(u16(ck)), orc.calibrate_per_head(u16(cv))
    orc.cache_write(mode, kb, vb, slots, kc, vc, ks, vs, k_scale=sk, v_scale=sv)
    L = w.context_lens[0]
    last = np.array([b * L + L - 1 for b in range(w.B)])
    q = u16(wl.queries(w, "cpu"))
    st = dict(w=w, pg=pg, kc=kc, vc=vc, ks=ks, vs=vs, sk=sk, sv=sv, q=q,
              kn=np.ascontiguousarray(kb[last]), vn=np.ascontiguousarray(vb[last]),
              sl=slots[last], bt=pg.block_table.numpy(), cl=pg.context_lens.numpy())
    return st


def oracle_step(mode: int, st) -> None:
    from oracle import oracle as orc
    orc.cache_write(mode, st["kn"], st["vn"], st["sl"], st["kc"], st["vc"], st["ks"], st["vs"],
                    k_scale=st["sk"], v_scale=st["sv"])
    orc.decode(mode, st["q"], st["kc"], st["vc"], st["bt"], st["cl"], k_scale=st["sk"],
               v_scale=st["sv"], k_cache_scale=st["ks"], v_cache_scale=st["vs"])


def cpu_baseline(args, mode: int, steps: int = 2):
    from oracle import oracle as orc
    n_seq = args.cpu_seqs
    st = oracle_step_setup(mode, n_seq)
    oracle_step(mode, st)
    t = time.perf_counter()
    for _ in range(steps):
        oracle_step(mode, st)
    dt = (time.perf_counter() - t) / steps
    w = st["w"]
    b = decode_bytes(w, mode) + write_bytes(w, mode, w.B)
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"{n_seq} of 64 sequences (x 4096 positions, all 32 heads) of the same "
                      f"decode step; {steps} timed steps of {dt:.2f} s wall each"}


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return None
    from oracle import oracle as orc
    from int4_quantized_paged_gb300.workloads import MODES
    mode = MODES[args.mode]
    st = oracle_step_setup(mode, args.cpu_seqs)
    for _ in range(args.warmup):
        oracle_step(mode, st)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(mode, st)
    dt = (time.perf_counter() - t) / args.steps
    w = st["w"]
    b = decode_bytes(w, mode) + write_bytes(w, mode, w.B)
    v = round(b / dt / 1e9, 4)
    sample = (f"{args.cpu_seqs} of 64 sequences (x 4096 positions, all 32 heads) of the "
              f"llama8b decode step, per step")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3" if mode in (1, 2, 3) else ("int4" if mode == 4 else "bf16"),
        "data": "synthetic", "config": {"workload": "llama8b-like decode step (sampled)",
                                        "mode": args.mode},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="fp8_per_token_head",
                    choices=["bf16", "fp8_per_tensor", "fp8_per_head", "fp8_per_token_head",
                             "int4_per_token_head"])
    ap.add_argument("--workers", type=int, default=0)
    ap.add_argument("--cpu-seqs", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
