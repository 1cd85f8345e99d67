"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1), no GPU.

The layer shards as independent replicas (every token is independent once the experts are
replicated), so the only cross-rank operations are the timing contract's barrier and the max over
ranks; the whole-job value is the replicas' tokens over the slowest rank's time.  The reference
arm under torchrun runs on rank 0 alone and the other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert torch.distributed.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")   # rank 1 is the slowest
    value = bench.replica_throughput(256, 4, w, slowest)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "value": value}, f)
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_barrier_max_and_value(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == 15.0                       # the max over ranks, seen by both
        assert r["value"] == pytest.approx(256 * 4 * 2 / 0.015)   # all replicas' tokens / slowest


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.replica_throughput(100, 10, 1, 1000.0) == pytest.approx(1000.0)


@pytest.mark.skipif(torch.cuda.is_available(), reason="the CPU (gloo) launch of the reference arm")
def test_reference_arm_under_torchrun_prints_once(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny_f32", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
