"""Host-side checks of the benchmark harness: replica timing aggregation over
a 2-rank gloo group on CPU, and the CPU-oracle reference arm's contract."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each replica reports its own step time; the job is as slow as the slowest
        out[rank] = bench.reduce_max(1.5 + rank, dist)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replica_timing_takes_the_max_over_ranks():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reduce_max_without_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25) == 3.25


def run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_quietly():
    r = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"],
                  {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line():
    r = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"],
                  {"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "resnet_3x3_64to128_56"


def test_warmup_below_three_is_refused():
    r = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "2"], {})
    assert r.returncode != 0


def test_source_hash_ignores_comments_only():
    """The traffic figure is tied to the kernel's code: comments and blank lines
    do not change the hash, any code edit does, and literals are left intact."""
    import bench
    src = ('// header\nint a = 1;  // trailing\n/* block\n   comment */\n\n'
           'const char* s = "a // b /* c */";\nchar q = \'/\';\nint b = 2; /* x */ int c = 3;\n')
    assert bench.strip_comments(src) == (
        'int a = 1;\nconst char* s = "a // b /* c */";\nchar q = \'/\';\nint b = 2;  int c = 3;')
    assert bench.strip_comments(src.replace("trailing", "other words")) == bench.strip_comments(src)
    assert bench.strip_comments(src.replace("int a = 1", "int a = 2")) != bench.strip_comments(src)
    assert len(bench.kernel_source_hash()) == 64


def test_sweep_summary_keeps_every_workload_and_stays_short():
    # the sweep entries of a recorded benchmark run, one per workload, as the
    # headline line carries them: every workload present, a few KB in all
    import json
    import bench
    import workloads
    full = []
    for i, c in enumerate(workloads.ALL):
        full.append({"workload": c.name, "path": "window", "us": 10.0 + i / 3, "tflops": 900.123456,
                     "gbs": 2000.5, "bound": "tensor", "roofline_us": 7.9, "frac_of_roofline": 0.5123456,
                     "workspace_bytes": 0, "im2col_bytes": 115605504, "im2win_bytes": 1,
                     "gemm_kernel_us": 9.9, "gemm_frac_of_roofline": 0.6, "im2win_us": 5.0,
                     "im2win_gbs": 2528.8, "im2win_frac_hbm": 0.37})
    full[3] = {"workload": workloads.ALL[3].name, "error": "x" * 300}
    s = bench.sweep_summary(full)
    assert list(s) == [c.name for c in workloads.ALL]
    assert s[workloads.ALL[0].name] == {"path": "window", "us": 10.0, "tflops": 900.1, "frac": 0.512,
                                        "bound": "tensor", "ws_B": 0}
    assert len(s[workloads.ALL[3].name]["error"]) == 80
    assert len(json.dumps(s)) < 3000 < len(json.dumps(full))
