"""The N > 1 path of bench.py on CPU: two gloo ranks.

bench.py runs one independent replica per GPU (the path has no exchange
step), so the multi-rank logic is host-side: the timed region is the
slowest rank's, the reported value counts the blocks of all ranks, and the
reference arm prints from rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [0.25, 0.75][rank]                      # rank 1 is the slower one
    secs = bench.max_over_ranks(local, world, "cpu")
    value = bench.whole_job_value(world, 100, secs)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"secs": secs, "value": value}, f)


def test_slowest_rank_sets_the_time_and_all_ranks_count(tmp_path):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for g in got:
        assert g["secs"] == 0.75
        assert g["value"] == pytest.approx(2 * 100 / 0.75)


def test_single_rank_passes_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1, "cpu") == 0.5
    assert bench.whole_job_value(1, 10, 2.0) == 5.0


def test_reference_arm_prints_once_under_torchrun(tmp_path):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-rows", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
