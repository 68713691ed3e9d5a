"""Benchmark of the quantized paged KV cache hot path on one GB300.

One step = one decode step of the 70B-like long-context layer (Hq=64, Hkv=8,
D=128, block 16, batch 8 x context 131072, dynamic per-token-head FP8 by
default): kvq_cache_write of the current token of every sequence, then
kvq_decode_attention (split-K over the 131,072 cached positions, log-sum-exp
merge).  Throughput is algorithmic bytes (what the method must move: codes,
scales, q, out, block table, new K/V and slots) per second.  The same run
also times a prefill-shaped cache write of the whole 1,048,576-token context
(cache-write GB/s), and then measures every other workload and mode the same
way (the "configs" block: decode and fill GB/s and their fractions of the
measured HBM peak, per-kernel CUDA-event times) and a few prefill chunks (the
"prefill" block: TFLOP/s against the tensor peak).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode fp8_per_token_head]
                    [--workload llama70b_128k|llama8b|gptoss20b|gemma_d256]
                    [--skip-sliding] [--workers N] [--graph | --no-graph] [--no-configs]
                    [--no-prefill]
                    [--batch B] [--context L] [--layer I]     # smaller cases (profiling)
    python bench.py --impl reference     # the CPU oracle on a bounded sample
    python bench.py --prefill --workload llama8b|gemma_d256|gptoss20b     # prefill TFLOP/s
    python bench.py --latency-sweep --workload gptoss20b        # latency vs context

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
work shards by sequence with no exchange); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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


def measured_peak(names, path=None):
    """First positive number stored under one of `names` anywhere in the
    measured-peaks file (top level or nested), else None."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None

    def find(node, name):
        if isinstance(node, dict):
            v = node.get(name)
            if isinstance(v, (int, float)) and not isinstance(v, bool) and v > 0:
                return float(v)
            for child in node.values():
                r = find(child, name)
                if r is not None:
                    return r
        elif isinstance(node, list):
            for child in node:
                r = find(child, name)
                if r is not None:
                    return r
        return None

    for name in names:
        r = find(d, name)
        if r is not None:
            return r
    return None


def peak_hbm(path=None):
    """HBM copy bandwidth (GB/s) and its source."""
    v = measured_peak(("hbm_gbs", "hbm_GBps"), path)
    return (v, "measured") if v else (FALLBACK_HBM_GBS, "fallback")


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
WORKLOADS = {
    "llama8b": "llama8b-like decode step: Hq=32 Hkv=8 D=128 block 16, batch 64 x context 4096, "
               "1 layer, 1 query/seq",
    "llama70b_128k": "70B-like long-context decode step: Hq=64 Hkv=8 D=128 block 16, batch 8 x "
                     "context 131072, 1 layer",
    "gptoss20b": "gpt-oss-20b-like 24-layer decode step: layers alternate window 128 / full, Hq=64 "
                 "Hkv=8 D=64 block 16, batch 16 x context 32768",
    "gemma_d256": "Gemma-like decode step: 2 layers (window 512, full), Hq=16 Hkv=8 D=256 block "
                  "16, batch 32 x context 16384",
}


def rank_workload(name: str, rank: int, args=None):
    """The workload a rank runs: the same shapes, its own seed (the path
    shards by sequence, so each replica draws its own batch).  --batch,
    --context and --layer shrink it (small cases for profiler captures)."""
    import dataclasses
    from int4_quantized_paged_gb300 import workloads as wl
    base = wl.CONFIGS[name]
    w = dataclasses.replace(base, seed=base.seed + 1000 * rank)
    if args is not None and (getattr(args, "batch", 0) or getattr(args, "context", 0)):
        w = wl.scaled(w, batch=args.batch or None, context=args.context or None)
    if args is not None and getattr(args, "layer", None) is not None:
        w = dataclasses.replace(w, windows=(w.windows[args.layer],))
    return w


def shape_note(args) -> str:
    """Text appended to the workload description when the shape was shrunk."""
    parts = []
    if getattr(args, "batch", 0):
        parts.append(f"batch {args.batch}")
    if getattr(args, "context", 0):
        parts.append(f"context {args.context}")
    if getattr(args, "layer", None) is not None:
        parts.append(f"layer {args.layer} only")
    return f" [reduced: {', '.join(parts)}]" if parts else ""


def layer_modes(w, mode: int, skip_sliding: bool):
    """Per-layer cache mode: the chosen mode, or BF16 for window layers when
    the sliding layers are skipped."""
    return [0 if (skip_sliding and win > 0) else mode for win in w.windows]


def setup_gpu(args, dev, rank, w=None, time_fill=True):
    """Caches of every layer filled with the context minus the current token,
    the step's inputs, workspaces.  Returns a dict of state."""
    import torch
    from int4_quantized_paged_gb300 import kvq
    from int4_quantized_paged_gb300 import workloads as wl

    w = rank_workload(args.workload, rank, args) if w is None else w
    L = w.context_lens[0]
    modes = layer_modes(w, kvq.MODE_NAMES[args.mode], args.skip_sliding)
    pg = wl.paging(w, dev)
    ctx = kvq.kvq_create(w.num_layers, w.Hq, w.Hkv, w.D, w.block_size, pg.num_blocks, modes,
                         list(w.windows))
    layers = []
    fill_ms = None
    for li, (mode, win) in enumerate(zip(modes, w.windows)):
        kc, vc, ks, vs = kvq.alloc_layer_cache(ctx, li, dev)
        k_scale = v_scale = None
        if mode == kvq.FP8_PER_TENSOR:
            k_scale = torch.ones(1, device=dev)
            v_scale = torch.ones(1, device=dev)
        elif mode == kvq.FP8_PER_HEAD:
            ck, cv = wl.calibration_sample(w, dev, layer=li)
            k_scale = torch.empty(w.Hkv, device=dev)
            v_scale = torch.empty(w.Hkv, device=dev)
            kvq.kvq_calibrate_per_head(ctx, ck, k_scale)
            kvq.kvq_calibrate_per_head(ctx, cv, v_scale)
        # fill: every retained position but the current one
        lo = max(0, L - win) if win > 0 else 0
        pos = [torch.arange(lo, L, dtype=torch.int64) for _ in range(w.B)]
        T = sum(len(p) for p in pos)
        k_all, v_all = wl.kv_tokens(w, T, dev, layer=li)
        slots_all = wl.slot_mapping(w, pg, pos, dev)

        def fill():
            kvq.kvq_cache_write(ctx, li, k_all, v_all, slots_all, kc, vc, ks, vs, k_scale, v_scale)

        fill()
        if time_fill and fill_ms is None and win == 0:
            # prefill-shaped write of the whole context of one full layer
            for _ in range(3):
                fill()
            torch.cuda.synchronize()
            ts = []
            stream = torch.cuda.current_stream()
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fill()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            fill_ms = (statistics.median(ts), T, mode)
        n_per = L - lo
        idx = torch.tensor([b * n_per + n_per - 1 for b in range(w.B)], device=dev)
        k_new, v_new = k_all[idx].contiguous(), v_all[idx].contiguous()
        del k_all, v_all, slots_all
        q = wl.queries(w, dev, layer=li)
        out = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32, device=dev)
        workers, ws_bytes = kvq.kvq_decode_plan(ctx, li, w.B, L, args.workers)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        layers.append(dict(mode=mode, window=win, kc=kc, vc=vc, ks=ks, vs=vs, k_scale=k_scale,
                           v_scale=v_scale, k_new=k_new, v_new=v_new, q=q, out=out,
                           workers=workers, ws=ws))
    slots_new = wl.slot_mapping(w, pg, [torch.tensor([L - 1]) for _ in range(w.B)], dev)
    torch.cuda.synchronize()
    return dict(w=w, L=L, pg=pg, ctx=ctx, layers=layers, slots_new=slots_new, fill=fill_ms)


def launch_layer(st, li, ev=None, stream=None, inputs=None, out=None):
    """One layer of the decode step: write the current token, then decode."""
    from int4_quantized_paged_gb300 import kvq
    lay = st["layers"][li]
    out = lay["out"] if out is None else out
    q, kn, vn, sl, bt, cl = inputs if inputs is not None else (
        lay["q"], lay["k_new"], lay["v_new"], st["slots_new"], st["pg"].block_table,
        st["pg"].context_lens)
    if ev is not None:
        ev[0].record(stream)
    kvq.kvq_cache_write(st["ctx"], li, kn, vn, sl, lay["kc"], lay["vc"], lay["ks"], lay["vs"],
                        lay["k_scale"], lay["v_scale"])
    if ev is not None:
        ev[1].record(stream)
    kvq.kvq_decode_attention(st["ctx"], li, q, lay["kc"], lay["vc"], bt, cl, out,
                             max_context=st["L"], k_scale=lay["k_scale"], v_scale=lay["v_scale"],
                             k_cache_scale=lay["ks"], v_cache_scale=lay["vs"],
                             num_workers=lay["workers"], workspace=lay["ws"])
    if ev is not None:
        ev[2].record(stream)


def layer_breakdown(layers, dbytes, dec_ms, write_ms):
    """Per-layer times of the step (mean CUDA-event ms of each layer's write
    and decode + merge) and the decode's algorithmic GB/s, layers in order."""
    out = []
    for li, lay in enumerate(layers):
        d = statistics.mean(dec_ms[li])
        out.append({"layer": li, "mode": int(lay["mode"]), "window": int(lay["window"]),
                    "decode_ms": round(d, 5),
                    "decode_gbs": round(dbytes[li] / (d * 1e-3) / 1e9, 2) if d > 0 else None,
                    "write_ms": round(statistics.mean(write_ms[li]), 5)})
    return out


def run_gpu(args):
    import torch
    from int4_quantized_paged_gb300 import kvq

    rank, world, local = rank_env()
    torch.cuda.set_device(local)
    dist = init_dist("nccl")
    dev = f"cuda:{local}"
    st = setup_gpu(args, dev, rank)
    w, L, layers = st["w"], st["L"], st["layers"]
    nl = len(layers)
    stream = torch.cuda.current_stream()
    use_graph = args.graph if args.graph is not None else nl > 1

    def step():
        for li in range(nl):
            launch_layer(st, li)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kvq.kvq_get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # per-kernel times: un-graphed steps with events around each launch
    n_ev = min(args.steps, 200) if args.steps > 0 else 200
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nl)]
          for _ in range(n_ev if not use_graph else min(n_ev, 10))]
    torch.cuda.synchronize()
    for i in range(len(ev)):
        for li in range(nl):
            launch_layer(st, li, ev[i][li], stream)
    torch.cuda.synchronize()
    write_ms = [[ev[i][li][0].elapsed_time(ev[i][li][1]) for i in range(len(ev))] for li in range(nl)]
    dec_ms = [[ev[i][li][1].elapsed_time(ev[i][li][2]) for i in range(len(ev))] for li in range(nl)]
    # --steps 0: enough steps for about a second of timed work, so that the
    # clock samples (every 200 ms) fall inside the loaded region
    est_ms = sum(statistics.mean(x) for x in write_ms) + sum(statistics.mean(x) for x in dec_ms)
    n = args.steps if args.steps > 0 else int(min(20000, max(50, math.ceil(1000.0 / est_ms))))

    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream()
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            step()                                # warm the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=s2):
                step()
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()

    # the timed region
    sampler = ClockSampler(local)
    sampler.start()
    t_pre = time.time()
    while time.time() - t_pre < 0.4:      # keep the GPU loaded while the sampler starts
        for _ in range(max(1, n // 4)):
            graph.replay() if graph is not None else step()
        torch.cuda.synchronize()
    barrier(dist, local)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(n):
        if graph is not None:
            graph.replay()
        else:
            step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, local)
    total_ms = t0.elapsed_time(t1)
    clocks = sampler.stop()
    if kvq.kvq_get_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")

    # end to end through the C ABI with host buffers (un-graphed calls): the
    # step's inputs travel in one pinned staging buffer (one host-to-device
    # copy) and its outputs come back in one (one device-to-host copy); the
    # kernels read and write views of the device-side buffers
    def layout(tensors):
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, total

    in_t = [st["slots_new"], st["pg"].block_table, st["pg"].context_lens] + \
        [lay[k] for lay in layers for k in ("q", "k_new", "v_new")]
    offs, total_in = layout(in_t)
    h_in = torch.empty(total_in, dtype=torch.uint8).pin_memory()
    for t, o in zip(in_t, offs):
        nb = t.numel() * t.element_size()
        h_in[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    d_in = torch.empty(total_in, dtype=torch.uint8, device=dev)
    dv = [d_in[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
          for t, o in zip(in_t, offs)]
    out_t = [lay["out"] for lay in layers]
    ooffs, total_out = layout(out_t)
    d_out = torch.empty(total_out, dtype=torch.uint8, device=dev)
    ov = [d_out[o:o + t.numel() * 4].view(torch.float32).view(t.shape)
          for t, o in zip(out_t, ooffs)]
    h_out = torch.empty(total_out, dtype=torch.uint8).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in in_t)
    d2h = sum(t.numel() * t.element_size() for t in out_t)

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        for li in range(nl):
            q, kn, vn = dv[3 + 3 * li:6 + 3 * li]
            launch_layer(st, li, inputs=(q, kn, vn, dv[0], dv[1], dv[2]), out=ov[li])
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist, local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n

    # ---- numbers
    ms_step = max_over_ranks(dist, total_ms / n)
    e2e_ms = max_over_ranks(dist, e2e_ms)
    dbytes = [decode_bytes(w, lay["mode"], lay["window"]) for lay in layers]
    wbytes = [write_bytes(w, lay["mode"], w.B) for lay in layers]
    step_bytes = sum(dbytes) + sum(wbytes)
    all_bytes = sum_over_ranks(dist, step_bytes)
    kv_pos = sum(sum(min(Lb, lay["window"]) if lay["window"] else Lb for Lb in w.context_lens)
                 for lay in layers)
    kv_tokens = sum_over_ranks(dist, float(kv_pos))
    peak, peak_src = peak_hbm()
    # dominant kernel: the decode of the layer with the most algorithmic bytes
    top = max(range(nl), key=lambda li: dbytes[li] * 1e6 + li)
    dec_avg = statistics.mean(dec_ms[top])
    dec_gbs = dbytes[top] / (dec_avg * 1e-3) / 1e9
    fill_ms, fill_T, fill_mode = st["fill"]
    wb_fill = write_bytes(w, fill_mode, fill_T)
    fill_gbs = wb_fill / (fill_ms * 1e-3) / 1e9
    summary = f"decode_{args.workload}_{args.mode}.md"
    traffic = profiled_traffic("decode.cu", summary)
    mode_name = args.mode + ("+bf16_sliding" if args.skip_sliding else "")
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
        "dtype": {0: "bf16", 4: "int4"}.get(layers[top]["mode"], "fp8_e4m3"),
        "data": "synthetic (seeded; N(0,1) with the workload's per-head multipliers and outliers)",
        "config": {"workload": WORKLOADS[args.workload] + shape_note(args), "mode": mode_name,
                   "num_workers": layers[top]["workers"], "cuda_graph": bool(graph is not None),
                   "l2": "inputs larger than L2: %.0f MB of cache read per step vs 129 MB L2"
                         % (sum(dbytes) / 1e6),
                   "parallelism": f"replicas x{world} (no exchange)"},
        "kv_tokens_per_s": round(kv_tokens / (ms_step * 1e-3), 1),
        "decode": {"gbs": round(dec_gbs, 2), "ms": round(dec_avg, 5), "layer": top,
                   "bytes_per_launch": dbytes[top], "frac_of_peak": round(dec_gbs / peak, 4)},
        "write_step": {"gbs": round(sum(wbytes) / (sum(statistics.mean(x) for x in write_ms) * 1e-3) / 1e9, 2),
                       "ms": round(sum(statistics.mean(x) for x in write_ms), 5),
                       "tokens": w.B * nl},
        "write_fill": {"gbs": round(fill_gbs, 2), "ms": round(fill_ms, 4), "tokens": fill_T,
                       "bytes": wb_fill, "frac_of_peak": round(fill_gbs / peak, 4)},
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "kernel": "decode_kernel (+ log-sum-exp merge)",
                     "peak_source": f"{peak_src} hbm_gbs",
                     "traffic_source": (f"profiles/{summary}: ncu dram bytes per launch, "
                                        "captured on the same decode.cu (sha256 checked), "
                                        "not measured in this run") if traffic else None},
        "e2e": {"value": round(all_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5)},
        "layers": layer_breakdown(layers, dbytes, dec_ms, write_ms),
        # per layer: the write, the decode and (with more than one worker) the merge
        "gpu_launches": n * sum(3 if lay["workers"] > 1 else 2 for lay in layers),
        "clocks": clocks,
    }
    del st, layers, d_in, d_out, dv, ov
    if graph is not None:
        del graph
    torch.cuda.empty_cache()
    if world == 1 and not args.no_configs:
        res["configs"] = config_block(args, dev)
    if world == 1 and not args.no_prefill:
        res["prefill"] = prefill_block(args)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args, kvq.MODE_NAMES[args.mode])
    if dist is not None:
        dist.destroy_process_group()
    return res if rank == 0 else None


# Every configuration of the five workloads that has a roofline target, each
# measured in the same run as the headline: (workload, mode, skip sliding).
CONFIG_BLOCK = [
    ("llama8b", "fp8_per_tensor", False),
    ("llama8b", "fp8_per_head", False),
    ("llama8b", "fp8_per_token_head", False),
    ("llama8b", "int4_per_token_head", False),
    ("llama70b_128k", "fp8_per_tensor", False),
    ("llama70b_128k", "fp8_per_head", False),
    ("llama70b_128k", "fp8_per_token_head", False),
    ("gptoss20b", "fp8_per_token_head", False),
    ("gptoss20b", "fp8_per_token_head", True),
    ("gemma_d256", "fp8_per_token_head", False),
    ("gemma_d256", "int4_per_token_head", False),
]


def measure_config(args, dev, workload: str, mode: str, skip: bool, steps: int = 20) -> dict:
    """One configuration's decode step, timed kernel by kernel with CUDA events
    on the launching stream, plus its prefill-shaped fill of one full layer.
    Decode GB/s is the largest layer's decode (+ merge) launch: its
    algorithmic bytes / its mean event time; the step is the whole write +
    decode of every layer (a CUDA graph for multi-layer workloads)."""
    import types
    import torch
    from int4_quantized_paged_gb300 import kvq
    a = types.SimpleNamespace(**{**vars(args), "workload": workload, "mode": mode,
                                 "skip_sliding": skip, "batch": 0, "context": 0, "layer": None,
                                 "workers": 0})
    st = setup_gpu(a, dev, 0)
    w, layers = st["w"], st["layers"]
    nl = len(layers)
    stream = torch.cuda.current_stream()

    def step():
        for li in range(nl):
            launch_layer(st, li)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nl)]
          for _ in range(steps)]
    for i in range(steps):
        for li in range(nl):
            launch_layer(st, li, ev[i][li], stream)
    torch.cuda.synchronize()
    write_ms = [statistics.mean(ev[i][li][0].elapsed_time(ev[i][li][1]) for i in range(steps))
                for li in range(nl)]
    dec_ms = [statistics.mean(ev[i][li][1].elapsed_time(ev[i][li][2]) for i in range(steps))
              for li in range(nl)]
    graph = None
    if nl > 1:
        graph = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream()
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            step()
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=s2):
                step()
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        graph.replay() if graph is not None else step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms_step = t0.elapsed_time(t1) / steps
    if kvq.kvq_get_device_error() != 0:
        raise RuntimeError(f"device error word set while measuring {workload} {mode}")
    peak, _ = peak_hbm()
    dbytes = [decode_bytes(w, lay["mode"], lay["window"]) for lay in layers]
    wbytes = [write_bytes(w, lay["mode"], w.B) for lay in layers]
    top = max(range(nl), key=lambda li: dbytes[li] * 1e6 + li)
    dec_gbs = dbytes[top] / (dec_ms[top] * 1e-3) / 1e9
    fill_ms, fill_T, fill_mode = st["fill"]
    wb_fill = write_bytes(w, fill_mode, fill_T)
    fill_gbs = wb_fill / (fill_ms * 1e-3) / 1e9
    kv_pos = sum(sum(min(Lb, lay["window"]) if lay["window"] else Lb for Lb in w.context_lens)
                 for lay in layers)
    out = {"workload": workload, "mode": mode + ("+bf16_sliding" if skip else ""),
           "layers": nl, "num_workers": layers[top]["workers"],
           "decode": {"bytes_per_launch": dbytes[top], "ms": round(dec_ms[top], 5),
                      "gbs": round(dec_gbs, 2), "frac_of_peak": round(dec_gbs / peak, 4)},
           "write_fill": {"bytes": wb_fill, "ms": round(fill_ms, 5), "tokens": fill_T,
                          "gbs": round(fill_gbs, 2), "frac_of_peak": round(fill_gbs / peak, 4)},
           "write_step_ms": round(sum(write_ms), 5),
           "decode_step_ms": round(sum(dec_ms), 5),
           "step": {"ms": round(ms_step, 5), "cuda_graph": graph is not None,
                    "gbs": round((sum(dbytes) + sum(wbytes)) / (ms_step * 1e-3) / 1e9, 2),
                    "kv_tokens_per_s": round(kv_pos / (ms_step * 1e-3), 1)}}
    del st, graph
    torch.cuda.empty_cache()
    return out


def config_block(args, dev) -> list:
    return [measure_config(args, dev, wname, mode, skip) for wname, mode, skip in CONFIG_BLOCK]


# Prefill chunks timed after the decode configurations (kvq_prefill_attention;
# TFLOP/s against the tensor peak), so the default run records the prefill
# kernels too: (workload, mode).
PREFILL_BLOCK = [
    ("llama8b", "fp8_per_token_head"),
    ("llama8b", "fp8_per_head"),
    ("llama8b", "int4_per_token_head"),
    ("llama8b", "bf16"),
    ("gemma_d256", "fp8_per_token_head"),
    ("gptoss20b", "fp8_per_token_head"),
]


def prefill_block(args) -> list:
    out = []
    for wname, mode in PREFILL_BLOCK:
        sub = argparse.Namespace(workload=wname, mode=mode, steps=5, warmup=3)
        r = run_prefill(sub)
        out.append({"workload": wname, "mode": mode, "chunk": r["config"]["workload"],
                    "kernel": r["roofline"]["kernel"], "tflops": r["value"],
                    "frac_of_peak": r["roofline"]["frac"], "ms": r["ms_per_step"],
                    "tokens_per_s": r["config"]["tokens_per_s"]})
    return out


# ------------------------------------------------------------------ oracle arm
# CPU sample per workload: (sequences, KV heads with all their query heads)
CPU_SAMPLE = {"llama8b": (8, 8), "llama70b_128k": (1, 1), "gptoss20b": (1, 1), "gemma_d256": (1, 2)}


def oracle_step_setup(args, n_seq: int):
    """Bounded sample of the same workload for the CPU oracle: n_seq of its
    sequences and the first few KV heads (with all their query heads), every
    layer; caches written by the oracle (untimed)."""
    import numpy as np
    import torch
    from int4_quantized_paged_gb300 import workloads as wl
    from int4_quantized_paged_gb300.workloads import MODES
    from oracle import oracle as orc

    base = wl.CONFIGS[args.workload]
    n_seq = min(n_seq or CPU_SAMPLE[args.workload][0], base.B)
    n_kv = CPU_SAMPLE[args.workload][1]
    w = wl.Workload(**{**base.__dict__, "context_lens": base.context_lens[:n_seq]})
    modes = layer_modes(w, MODES[args.mode], args.skip_sliding)
    pg = wl.paging(w, "cpu")
    L = w.context_lens[0]
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    layers = []
    for li, (mode, win) in enumerate(zip(modes, w.windows)):
        lo = max(0, L - win) if win > 0 else 0
        pos = [torch.arange(lo, L, dtype=torch.int64) for _ in range(w.B)]
        T = sum(len(p) for p in pos)
        k, v = wl.kv_tokens(w, T, "cpu", layer=li)
        slots = wl.slot_mapping(w, pg, pos, "cpu").numpy()
        kb, vb = u16(k), u16(v)
        kc, vc, ks, vs = orc.alloc_cache(mode, pg.num_blocks, w.Hkv, w.block_size, w.D)
        sk = sv = None
        if mode == 1:
            sk = sv = np.ones(1, dtype=np.float32)
        elif mode == 2:
            ck, cv = wl.calibration_sample(base, "cpu", layer=li)
            sk, sv = orc.calibrate_per_head(u16(ck)), orc.calibrate_per_head(u16(cv))
        orc.cache_write(mode, kb, vb, slots, kc, vc, ks, vs, k_scale=sk, v_scale=sv)
        n_per = L - lo
        last = np.array([b * n_per + n_per - 1 for b in range(w.B)])
        layers.append(dict(mode=mode, window=win, kc=kc, vc=vc, ks=ks, vs=vs, sk=sk, sv=sv,
                           q=u16(wl.queries(w, "cpu", layer=li)),
                           kn=np.ascontiguousarray(kb[last]), vn=np.ascontiguousarray(vb[last]),
                           sl=slots[last]))
    pairs = [(b, g * w.G + j) for b in range(w.B) for g in range(n_kv) for j in range(w.G)]
    return dict(w=w, layers=layers, bt=pg.block_table.numpy(), cl=pg.context_lens.numpy(),
                pairs=pairs, n_kv=n_kv)


def oracle_step(st) -> None:
    from oracle import oracle as orc
    for lay in st["layers"]:
        orc.cache_write(lay["mode"], lay["kn"], lay["vn"], lay["sl"], lay["kc"], lay["vc"],
                        lay["ks"], lay["vs"], k_scale=lay["sk"], v_scale=lay["sv"])
        orc.decode(lay["mode"], lay["q"], lay["kc"], lay["vc"], st["bt"], st["cl"],
                   k_scale=lay["sk"], v_scale=lay["sv"], k_cache_scale=lay["ks"],
                   v_cache_scale=lay["vs"], window=lay["window"], pairs=st["pairs"])


def oracle_bytes(st) -> float:
    """Algorithmic bytes of the sampled items: decode of n_kv KV heads (and
    their query heads) of the sampled sequences, write of their new tokens."""
    import dataclasses
    w = st["w"]
    ws = dataclasses.replace(w, Hkv=st["n_kv"], Hq=st["n_kv"] * w.G)
    return sum(decode_bytes(ws, lay["mode"], lay["window"]) + write_bytes(w, lay["mode"], w.B)
               for lay in st["layers"])


def cpu_baseline(args, mode: int, seconds: float = 10.0):
    """Times the oracle on a bounded sample for about `seconds` of wall time
    (at least two steps)."""
    from oracle import oracle as orc
    st = oracle_step_setup(args, args.cpu_seqs)
    oracle_step(st)
    t = time.perf_counter()
    steps = 0
    while steps < 2 or time.perf_counter() - t < seconds:
        oracle_step(st)
        steps += 1
    dt = (time.perf_counter() - t) / steps
    # the same sample on one thread (two steps)
    n_all = orc.num_threads()
    orc.set_num_threads(1)
    try:
        t1 = time.perf_counter()
        for _ in range(2):
            oracle_step(st)
        dt1 = (time.perf_counter() - t1) / 2
    finally:
        orc.set_num_threads(n_all)
    w = st["w"]
    return {"value": round(oracle_bytes(st) / dt / 1e9, 4), "unit": "GB/s",
            "cores": n_all, "kind": "oracle",
            "value_one_thread": round(oracle_bytes(st) / dt1 / 1e9, 4),
            "sample": f"{w.B} of {wl_batch(args)} sequences x {st['n_kv']} of {w.Hkv} KV heads "
                      f"(their query heads, every layer) of the same decode step; {steps} timed "
                      f"steps of {dt:.2f} s wall each on {n_all} threads, 2 steps of "
                      f"{dt1:.2f} s on one"}


def wl_batch(args) -> int:
    from int4_quantized_paged_gb300 import workloads as wl
    return wl.CONFIGS[args.workload].B


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return None
    from oracle import oracle as orc
    from int4_quantized_paged_gb300.workloads import MODES
    mode = MODES[args.mode]
    st = oracle_step_setup(args, args.cpu_seqs)
    for _ in range(args.warmup):
        oracle_step(st)
    steps = args.steps if args.steps > 0 else 5
    t = time.perf_counter()
    for _ in range(steps):
        oracle_step(st)
    dt = (time.perf_counter() - t) / steps
    v = round(oracle_bytes(st) / dt / 1e9, 4)
    w = st["w"]
    sample = (f"{w.B} of {wl_batch(args)} sequences x {st['n_kv']} of {w.Hkv} KV heads (their "
              f"query heads, every layer) of the {args.workload} decode step, per step")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {0: "bf16", 4: "int4"}.get(mode, "fp8_e4m3"),
        "data": "synthetic", "config": {"workload": WORKLOADS[args.workload] + " (sampled)",
                                        "mode": args.mode},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def fit_line(points):
    """Least-squares line y = a + b x through (x, y) points: (a, b)."""
    n = len(points)
    mx = sum(x for x, _ in points) / n
    my = sum(y for _, y in points) / n
    sxx = sum((x - mx) ** 2 for x, _ in points)
    b = sum((x - mx) * (y - my) for x, y in points) / sxx if sxx > 0 else 0.0
    return my - b * mx, b


def break_even(a0, b0, a, b):
    """Context where the line a + b x meets the reference a0 + b0 x (None if
    they are parallel); below it the cheaper intercept wins, above it the
    smaller slope."""
    return None if b0 == b else (a - a0) / (b0 - b)


def run_latency_sweep(args):
    """Decode-step latency against context length for BF16, all-FP8, FP8 with
    BF16 window layers, and INT4 caches on one workload shape (batch fixed),
    with a least-squares line per variant (intercept, ms per context token)
    and the context at which each quantized variant breaks even with BF16.
    Each point is the median of CUDA-graph replays of the whole step (every
    layer: write of the current token, then decode)."""
    import types
    import torch
    from int4_quantized_paged_gb300 import workloads as wl

    dev = "cuda:0"
    torch.cuda.set_device(0)
    base = wl.CONFIGS[args.workload]
    contexts = [int(c) for c in args.sweep_contexts.split(",")]
    variants = [("bf16", "bf16", False), ("fp8", "fp8_per_token_head", False),
                ("fp8+bf16_sliding", "fp8_per_token_head", True),
                ("int4", "int4_per_token_head", False)]
    if not any(win > 0 for win in base.windows):
        variants = [v for v in variants if not v[2]]
    points = {name: [] for name, _, _ in variants}
    stream = torch.cuda.current_stream()
    for L in contexts:
        w = wl.scaled(base, context=L)
        for name, mode, skip in variants:
            a = types.SimpleNamespace(**{**vars(args), "mode": mode, "skip_sliding": skip})
            st = setup_gpu(a, dev, 0, w=w, time_fill=False)
            nl = len(st["layers"])

            def step():
                for li in range(nl):
                    launch_layer(st, li)

            for _ in range(3):
                step()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            s2 = torch.cuda.Stream()
            s2.wait_stream(stream)
            with torch.cuda.stream(s2):
                step()
                torch.cuda.synchronize()
                with torch.cuda.graph(graph, stream=s2):
                    step()
            torch.cuda.synchronize()
            reps = 10
            ts = []
            for _ in range(7):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    graph.replay()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) / reps)
            points[name].append((L, statistics.median(ts)))
            del st, graph
            torch.cuda.empty_cache()

    lines = {name: fit_line(p) for name, p in points.items()}
    a0, b0 = lines["bf16"]
    res = {"metric": "decode-step latency vs context (fitted ms per context token; break-even "
                     "context vs BF16)",
           "workload": WORKLOADS[args.workload], "batch": base.B, "contexts": contexts,
           "unit": "ms per step", "variants": {}}
    for name, (a, b) in lines.items():
        v = {"ms": [round(y, 4) for _, y in points[name]], "intercept_ms": round(a, 5),
             "slope_ms_per_token": float("%.4g" % b)}
        if name != "bf16":
            be = break_even(a0, b0, a, b)
            v["break_even_context"] = None if be is None else round(be, 1)
        res["variants"][name] = v
    return res


PREFILL = {
    "llama8b": ("llama8b-like prefill chunk: 4 sequences x 1024 new tokens after 3072 cached, "
                "Hq=32 Hkv=8 D=128", 4, 3072, 1024),
    "gemma_d256": ("Gemma-like prefill chunk: 8192 new tokens at positions [8192, 16384) of one "
                   "sequence, Hq=16 Hkv=8 D=256, full-attention layer", 1, 8192, 8192),
    "gptoss20b": ("gpt-oss-like prefill chunk: 4 sequences x 1024 new tokens after 3072 cached, "
                  "Hq=64 Hkv=8 D=64, full-attention layer", 4, 3072, 1024),
}


def peak_tensor(path=None):
    """Dense bf16 tensor peak (TFLOP/s, the burst figure: the prefill kernel
    is timed alone) and its source."""
    v = measured_peak(("bf16_tflops", "bf16_dense_tflops"), path)
    return (v, "measured") if v else (1900.0, "fallback")


def run_prefill(args):
    """Prefill attention (kvq_prefill_attention) on one chunk shape: time and
    TFLOP/s of the causal QK and PV products (4 D flop per query-key pair)."""
    import torch
    from int4_quantized_paged_gb300 import kvq
    from int4_quantized_paged_gb300 import workloads as wl

    if args.workload not in PREFILL:
        raise SystemExit(f"--prefill: no chunk shape for workload {args.workload}; "
                         f"choose one of {sorted(PREFILL)}")
    desc, B, prefix, chunk = PREFILL[args.workload]
    dev = "cuda:0"
    torch.cuda.set_device(0)
    base = wl.CONFIGS[args.workload]
    L = prefix + chunk
    w = wl.Workload(**{**base.__dict__, "context_lens": tuple([L] * B), "windows": (0,)})
    mode = kvq.MODE_NAMES[args.mode]
    pg = wl.paging(w, dev)
    ctx = kvq.kvq_create(1, w.Hq, w.Hkv, w.D, w.block_size, pg.num_blocks, [mode], [0])
    kc, vc, ks, vs = kvq.alloc_layer_cache(ctx, 0, dev)
    k_scale = v_scale = None
    if mode in (kvq.FP8_PER_TENSOR, kvq.FP8_PER_HEAD):
        k_scale = torch.ones(w.Hkv if mode == kvq.FP8_PER_HEAD else 1, device=dev)
        v_scale = k_scale.clone()
    for b in range(B):
        pos = [torch.tensor([], dtype=torch.int64)] * b + [torch.arange(L)]
        k, v = wl.kv_tokens(w, L, dev, stream_base=40 + b)
        kvq.kvq_cache_write(ctx, 0, k, v, wl.slot_mapping(w, pg, pos, dev), kc, vc, ks, vs,
                            k_scale, v_scale)
    T = B * chunk
    g = torch.Generator(device=dev).manual_seed(base.seed + 77)
    q = torch.randn(T, w.Hq, w.D, generator=g, device=dev).to(torch.bfloat16)
    qs = torch.arange(0, T + 1, chunk, dtype=torch.int32, device=dev)
    out = torch.empty(T, w.Hq, w.D, dtype=torch.float32, device=dev)

    def step():
        kvq.kvq_prefill_attention(ctx, 0, q, kc, vc, pg.block_table, qs, pg.context_lens, out,
                                  max_query_len=chunk, k_scale=k_scale, v_scale=v_scale,
                                  k_cache_scale=ks, v_cache_scale=vs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kvq.kvq_get_device_error() != 0:
        raise RuntimeError("device error word set during prefill warm-up")
    n = args.steps if args.steps > 0 else 10
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(0)
    sampler.start()
    t_pre = time.time()
    while time.time() - t_pre < 0.4:
        step()
        torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / n
    clocks = sampler.stop()
    pairs = B * w.Hq * sum(prefix + i + 1 for i in range(chunk))
    tflops = 4.0 * pairs * w.D / (ms * 1e-3) / 1e12
    peak, src = peak_tensor()
    return {"metric": "prefill attention TFLOP/s (causal QK and PV, 4 D flop per query-key pair)",
            "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": n,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {0: "bf16", 4: "int4"}.get(mode, "fp8_e4m3"), "data": "synthetic",
            "config": {"workload": desc, "mode": args.mode,
                       "tokens_per_s": round(T / (ms * 1e-3), 1)},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "kernel": ("prefill_ws_kernel (tcgen05, warp-specialised, P' f16 hi + lo "
                                    "in tensor memory)" if w.D in ((64, 128) if mode == kvq.BF16 else (64, 128, 256))
                                    else "prefill_tc_kernel (tcgen05, P' split in shared memory)"),
                         "peak_source": f"{src} bf16 dense"},
            "gpu_launches": n, "clocks": clocks}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="0: as many steps as take about one second")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="fp8_per_token_head",
                    choices=["bf16", "fp8_per_tensor", "fp8_per_head", "fp8_per_token_head",
                             "int4_per_token_head"])
    ap.add_argument("--workers", type=int, default=0)
    ap.add_argument("--workload", default="llama70b_128k", choices=sorted(WORKLOADS))
    ap.add_argument("--skip-sliding", action="store_true",
                    help="keep the window layers' caches in BF16 (layer skipping)")
    ap.add_argument("--graph", dest="graph", action="store_true", default=None,
                    help="replay the step as a CUDA graph (default: on for multi-layer steps)")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload at this batch instead of its own (0: its own)")
    ap.add_argument("--context", type=int, default=0,
                    help="run the workload at this context instead of its own (0: its own)")
    ap.add_argument("--layer", type=int, default=None,
                    help="run only this layer of the workload (its window and mode)")
    ap.add_argument("--cpu-seqs", type=int, default=0, help="0: the workload's default sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill chunks timed after the decode configurations")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the block that measures every workload and mode after the headline")
    ap.add_argument("--latency-sweep", action="store_true",
                    help="latency against context for BF16 / FP8 / FP8 + BF16 window layers / "
                         "INT4 instead of the throughput line")
    ap.add_argument("--sweep-contexts", default="1024,2048,4096,8192,16384,32768")
    ap.add_argument("--prefill", action="store_true",
                    help="prefill attention on the workload's chunk shape instead of the decode step")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    if args.latency_sweep:
        res = run_latency_sweep(args)
    elif args.prefill:
        res = run_prefill(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
