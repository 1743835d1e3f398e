"""The benchmark's multi-process path on the CPU: two gloo ranks.

bench.py runs one replica per GPU (the GEMM shards by output tiles with no
exchange); the job's time is the slowest rank's and its throughput counts
every rank's work.  These tests run that aggregation over two real gloo
processes, and the reference arm's rank rule (rank 0 alone runs and prints).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.DistCtx(world, backend="gloo", device="cpu")
    d.barrier()
    local_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
    value, t = bench.whole_job(d, 2.0e12, 4, local_ms)
    total = d.sum(1.0)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"value": value, "t": t, "sum": total, "world": d.world}, f)
    d.pg.destroy_process_group()


def test_whole_job_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    for r in range(2):
        got = json.loads((tmp_path / f"r{r}.json").read_text())
        assert got["world"] == 2 and got["sum"] == 2.0
        assert got["t"] == 15.0                    # max over ranks
        # 2 ranks x 4 steps x 2e12 FLOP in 15 ms
        assert got["value"] == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, cwd=ROOT, timeout=600)


def test_reference_arm_runs_on_rank_zero_only():
    args = ("--impl", "reference", "--workload", "tile_f16_128x128x64", "--steps", "2", "--warmup", "0",
            "--gpus", "2")
    r1 = _bench({"RANK": "1", "WORLD_SIZE": "2"}, *args)
    assert r1.returncode == 0, r1.stderr[-2000:]
    assert r1.stdout.strip() == ""
    r0 = _bench({"RANK": "0", "WORLD_SIZE": "2"}, *args)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_kernel_clock_from_trace_stamps():
    # the SM clock the bench reports for a traced launch: per CTA, cycles
    # between the clock64 stamps over nanoseconds between the globaltimer
    # stamps; CTAs that did not run (zero slots) are left out
    import numpy as np
    import torch
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    tr = torch.zeros((4, 10), dtype=torch.int64)
    for c, (ns, ghz) in enumerate([(30_000, 1.6), (31_000, 1.8), (29_000, 2.0)]):
        tr[c, 0], tr[c, 6] = 1_000_000, 1_000_000 + ns
        tr[c, 8], tr[c, 9] = 5_000, 5_000 + int(ns * ghz)
    got = bench.kernel_clock(tr)
    assert got["kernel_sm_mhz"] == 1800.0
    assert got["kernel_sm_mhz_range"] == [1600.0, 2000.0]
    assert bench.kernel_clock(torch.zeros((3, 10), dtype=torch.int64)) == {"kernel_sm_mhz": None,
                                                                           "kernel_sm_mhz_range": None}
    assert np.isfinite(got["kernel_sm_mhz"])
