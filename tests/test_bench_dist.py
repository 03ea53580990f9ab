"""The benchmark's multi-rank path on CPU: two ranks over gloo.

With one process per GPU, each rank runs an independent replica of the step
(no collective on the data path); the ranks meet only at the barriers around
the timed region and in the max-over-ranks reduction of the elapsed time, and
rank 0 alone prints.  Run here with the gloo backend on 127.0.0.1."""
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
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(None)
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank k took 10 + k ms for 3 steps of its own replica
    ms, value = bench.aggregate(3, 10.0 + rank, w)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"ms": ms, "value": value}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r in res:
        # every rank sees the slowest rank's time; the job did 2 x 3 steps in it
        assert r["ms"] == pytest.approx(11.0)
        assert r["value"] == pytest.approx(2 * 3 / 11e-3)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone times
    the oracle and prints one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_2k_256",
           "--steps", "1", "--warmup", "0", "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
