"""The multi-GPU path without GPUs: world-size-2 process groups on CPU (gloo).

The row operations shard over rows with no data exchange, so several GPUs run
independent replicas ("replicas only"): the only cross-rank steps are the
barrier and the max over ranks of the step time, and `value` is the whole-job
throughput.  These run here on the gloo backend; the reference arm under
torchrun prints from rank 0 alone."""

import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

from tests.conftest import ROOT  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    # each replica's step time differs; every rank must see the slowest
    ms = bench.max_over_ranks(1.0 + rank * 0.5, "cpu")
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump({"ms": ms, "gbs": bench.aggregate_gbs(world, 10**9, ms)}, fh)
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == 1.5  # the slower rank's time on every rank
        # two replicas of 1 GB each in 1.5 ms
        assert abs(g["gbs"] - 2 * 1e9 / 1.5e-3 / 1e9) < 1e-9


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.aggregate_gbs(1, 2 * 10**9, 2.0) == 1000.0


def test_reference_arm_under_torchrun_prints_from_rank_zero_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--ref-rows", "16", "--workload", "small_f32_256x1024"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_attention_reference_arm_prints_one_line():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--cpu-budget-s", "0.4", "--workload", "attn_causal_32x96x512x128"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["T"] == 512 and d["config"]["D"] == 128


def test_attention_flop_and_byte_counts():
    sys.path.insert(0, ROOT)
    import bench
    # 4 D flops per visible (query, key) pair: T (T + 1) / 2 pairs per head under the causal mask
    assert bench.attention_flops(1, 1, 4, 8, True) == 4 * 8 * 10
    assert bench.attention_flops(2, 3, 4, 8, False) == 4 * 8 * 16 * 6
    # one read of bf16 q, k, v and one write of the output (bf16 by default) and fp32 lse
    assert bench.attention_bytes(1, 1, 4, 8) == 3 * 32 * 2 + 32 * 2 + 4 * 4
    assert bench.attention_bytes(1, 1, 4, 8, out_bytes=4) == 3 * 32 * 2 + 32 * 4 + 4 * 4


def test_cpu_baseline_times_one_thread_and_all_cores():
    # the oracle baseline: its value on one host thread, and the same sample split
    # over every host core (a spawn pool) beside it
    sys.path.insert(0, ROOT)
    import bench
    from softmax_cross_entropy_online_gb300 import synthetic
    d = bench.cpu_baseline(synthetic.WORKLOADS["small_f32_256x1024"], 0.2)
    assert d["kind"] == "oracle" and d["cores"] == 1 and d["value"] > 0
    n = os.cpu_count() or 1
    if n > 1:
        a = d["all_cores"]
        assert a["cores"] == n and a["value"] > 0 and a["unit"] == d["unit"]


def test_rate_figures():
    sys.path.insert(0, ROOT)
    import bench
    # fp32 [256, 1024] forward+backward: ~2.1 MB, far below a few microseconds at
    # 6.8 TB/s, so launch latency bounds it; [32768, 4096] (1.07 GB) does not
    small = bench.algorithmic_bytes(256, 1024, 4, True)
    r = bench.rate_figures(1, 256, 0.005, 0.004, small, 6800.0)
    assert r["latency_bound"] and abs(r["us_per_call"] - 4.0) < 1e-12
    assert abs(r["rows_per_s"] - 256 / 5e-6) < 1e-3
    big = bench.algorithmic_bytes(32768, 4096, 4, True)
    r = bench.rate_figures(2, 32768, 0.18, 0.18, big, 6800.0)
    assert not r["latency_bound"] and abs(r["rows_per_s"] - 2 * 32768 / 0.18e-3) < 1


def test_linear_cpu_baseline_on_a_small_shape():
    sys.path.insert(0, ROOT)
    import bench
    from softmax_cross_entropy_online_gb300 import synthetic
    M, H, V = 64, 32, 96
    h, W, t = synthetic.make_linear_ce_inputs(M, H, V, seed=0)
    d = bench.linear_cpu_baseline(h, W, t, M, H, V, 0.05)
    assert d["kind"] == "oracle" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cores"] >= 1 and "rows of h" in d["sample"]


def test_linear_reference_arm_prints_one_line(monkeypatch, capsys):
    # the reference arm of the linear + CE workload on a small stand-in shape
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setitem(bench.LINEAR_SHAPES, "linear_ce_8192x4096x128256", (64, 32, 96))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--workload",
                                      "linear_ce_8192x4096x128256", "--steps", "2"])
    assert bench.main() == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["value"] == d["value"] and d["config"]["sample_rows"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
