"""Host-side paths of bench.py that need no GPU.

* The replica aggregation over ranks (one process per GPU, launched by torchrun): with
  two gloo ranks on the CPU, the step time is the slowest rank's and the value counts
  both ranks' work.
* The reference arm (the CPU oracle on a row sample): rank 0 prints one JSON line with
  the contract's keys; other ranks exit 0 without output.
"""
import json
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    value, ms = bench.aggregate(1e12, 1.0 + rank, world, dist, torch.device("cpu"))
    out[rank] = (value, ms)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    world = 2
    port = 29000 + os.getpid() % 1000
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        value, ms = out[rank]
        assert ms == 2.0  # the slower rank's step time
        assert abs(value - world * 1e12 / 2e-3 / 1e12) < 1e-9  # 1000 TFLOP/s


def run_bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_other_ranks_exit_silently():
    p = run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--workloads",
                  "f32_256", "--steps", "1", "--warmup", "3", "--ref-budget-s", "2")
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    p = run_bench({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, "--impl", "reference", "--workloads",
                  "f32_256", "--steps", "2", "--warmup", "3", "--ref-budget-s", "3")
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "TFLOP/s"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["value"] == rec["value"]
    assert rec["steps"] == 2 and rec["warmup"] == 3


def test_clock_summary_counts_loaded_samples_and_reasons():
    sys.path.insert(0, ROOT)
    import bench
    idle = ["0", "1980", "2070", "120.5", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    busy = ["0", "1750", "2070", "1350.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    fast = ["0", "2070", "2070", "900.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    c = bench.summarize_clocks([idle, busy, busy, fast, idle])
    assert c["samples"] == 3 and c["sm_mhz"] == 1750.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and not bench.clocks_rejected(c)
    hot = list(busy)
    hot[7] = "Active"
    assert bench.clocks_rejected(bench.summarize_clocks([hot]))
    assert bench.summarize_clocks(None)["samples"] == 0
    assert bench.summarize_clocks([])["samples"] == 0


def test_fp32_peak_uses_the_given_sm_count():
    sys.path.insert(0, ROOT)
    import bench
    assert abs(bench.fp32_simt_peak_tflops(2070.0, 152) - 80.547) < 1e-3
    assert abs(bench.fp32_simt_peak_tflops(2070.0, 76) - 80.547 / 2) < 1e-3
