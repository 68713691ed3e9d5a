"""Host logic of the N > 1 benchmark path on CPU: two gloo ranks.

The path shards by sequence (replicas only, no data-path collective); what
the ranks share is the timing protocol: a barrier around the timed region,
the maximum of the ranks' step times and the sum of their bytes.
"""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.init_dist("gloo")
    r, ws, lr = bench.rank_env()
    bench.barrier(d)
    mx = bench.max_over_ranks(d, 1.5 + rank)          # step times 1.5 and 2.5 ms
    sm = bench.sum_over_ranks(d, 100.0 * (rank + 1))  # bytes 100 and 200
    w = bench.rank_workload("llama8b", rank)
    out[rank] = (r, ws, lr, mx, sm, w.seed)
    d.destroy_process_group()


def test_two_gloo_ranks_reduce_times_and_bytes():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    r0, r1 = out[0], out[1]
    assert (r0[0], r0[1], r0[2]) == (0, 2, 0) and (r1[0], r1[1], r1[2]) == (1, 2, 1)
    assert r0[3] == r1[3] == 2.5                      # max over ranks
    assert r0[4] == r1[4] == 300.0                    # sum over ranks
    assert r0[5] != r1[5]                             # each replica draws its own batch


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (0, 1, 0)
    assert bench.init_dist("gloo") is None
    assert bench.max_over_ranks(None, 3.0) == 3.0 and bench.sum_over_ranks(None, 4.0) == 4.0


def test_byte_accounting_matches_the_pages_per_token_formulas():
    # decode bytes of one full layer: positions x Hkv x (2 D elem + 8) + q + out + table
    from int4_quantized_paged_gb300 import workloads as wl
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=2, context=64)
    b = bench.decode_bytes(w, 3)
    assert b == 2 * 64 * 8 * (256 + 8) + 2 * 4 * 4 + 2 * 32 * 128 * 6
    assert bench.decode_bytes(w, 2) == 2 * 64 * 8 * 256 + 2 * 4 * 4 + 2 * 32 * 128 * 6
    assert bench.decode_bytes(w, 0, window=16) == 2 * 16 * 8 * 512 + 2 * 4 * 4 + 2 * 32 * 128 * 6
    # write bytes per token: Hkv x (bf16 K+V in + codes out + scales) + int64 slot
    assert bench.write_bytes(w, 3, 1) == 8 * (4 * 128 + 2 * 128 + 8) + 8 == 6216
    assert bench.write_bytes(w, 4, 1) == 8 * (4 * 128 + 128 + 8) + 8


def test_latency_sweep_line_fit_and_break_even():
    import bench
    pts = [(1024, 0.5 + 2e-5 * 1024), (4096, 0.5 + 2e-5 * 4096), (32768, 0.5 + 2e-5 * 32768)]
    a, b = bench.fit_line(pts)
    assert abs(a - 0.5) < 1e-12 and abs(b - 2e-5) < 1e-15
    # quantized line: higher intercept, lower slope -> meets BF16 at (0.6 - 0.5) / (3e-5 - 2e-5)
    assert abs(bench.break_even(0.5, 3e-5, 0.6, 2e-5) - 10000.0) < 1e-6
    assert bench.break_even(0.5, 2e-5, 0.6, 2e-5) is None


def test_reference_arm_prints_the_contract_line(capsys):
    """bench.py --impl reference runs the oracle on host cores and prints one
    JSON line with the keys the benchmark contract names."""
    import json
    import bench
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-seqs", "1"])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_under_torchrun_prints_once():
    """Launched as two ranks (the N > 1 form), the reference arm runs on rank 0
    only and prints exactly one line; the other rank exits 0."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29531", "bench.py", "--gpus", "2",
           "--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-seqs", "1"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_measured_peaks_read_flat_or_nested(tmp_path):
    """The roofline denominators come from the measured-peaks file whether
    its figures sit at the top level or inside a nested object; a missing or
    unreadable file falls back and says so."""
    flat = tmp_path / "flat.json"
    flat.write_text(json.dumps({"hbm_gbs": 6784.5, "bf16_tflops": 1936.0,
                                "bf16_tflops_sustained": 1700.0}))
    assert bench.peak_hbm(str(flat)) == (6784.5, "measured")
    assert bench.peak_tensor(str(flat)) == (1936.0, "measured")
    nested = tmp_path / "nested.json"
    nested.write_text(json.dumps({"gpu": "GB300", "peaks": {"hbm_gbs": 6700, "bf16_tflops": 1900.5}}))
    assert bench.peak_hbm(str(nested)) == (6700.0, "measured")
    assert bench.peak_tensor(str(nested)) == (1900.5, "measured")
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    assert bench.peak_hbm(str(bad)) == (bench.FALLBACK_HBM_GBS, "fallback")
    assert bench.peak_hbm(str(tmp_path / "absent.json"))[1] == "fallback"
    assert bench.peak_tensor(str(tmp_path / "absent.json")) == (1900.0, "fallback")


def test_layer_breakdown_reports_every_layer():
    """Per-layer decode and write times (a two-layer window / full pair)."""
    layers = [{"mode": 3, "window": 512}, {"mode": 3, "window": 0}]
    dbytes = [68.2e6, 2.18e9]
    dec_ms = [[0.02, 0.02], [0.33, 0.35]]
    write_ms = [[0.008], [0.009]]
    rows = bench.layer_breakdown(layers, dbytes, dec_ms, write_ms)
    assert [r["layer"] for r in rows] == [0, 1]
    assert [r["window"] for r in rows] == [512, 0]
    assert rows[0]["decode_gbs"] == round(68.2e6 / 0.02e-3 / 1e9, 2)
    assert rows[1]["decode_ms"] == 0.34 and rows[1]["write_ms"] == 0.009
    json.dumps(rows)


def test_bench_blocks_name_known_workloads_and_modes():
    """Every configuration and prefill chunk the default bench times names a
    workload the bench knows and a mode the library has, so the default line
    cannot fail on a misspelt entry."""
    from int4_quantized_paged_gb300.workloads import CONFIGS, MODES
    assert bench.CONFIG_BLOCK and bench.PREFILL_BLOCK
    for wname, mode, skip in bench.CONFIG_BLOCK:
        assert wname in bench.WORKLOADS and wname in CONFIGS, wname
        assert mode in MODES, mode
        assert isinstance(skip, bool)
    for wname, mode in bench.PREFILL_BLOCK:
        assert wname in bench.PREFILL and wname in CONFIGS, wname
        assert mode in MODES, mode
