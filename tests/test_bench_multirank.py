"""The N > 1 path of bench.py on CPU (gloo, world size 2): the max-over-ranks
time reduction, the per-rank shards, and a torchrun launch of the reference
arm (rank 0 alone prints one line; the other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        shards = bench.shard_configs(rank)
        q.put((rank, got, shards["c5_long_32k"]["seed"], shards["c5_long_32k"]["B"]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_shards_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]          # every rank sees the slowest time
    assert res[0][2] != res[1][2] and res[0][3] == res[1][3]  # distinct data, same shape


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5


def test_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "c1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("args", [["--workload", "c5", "--streams", "2"], ["--workload", "c3", "--streams", "0"]])
def test_streams_option_is_checked_before_any_work(args):
    """--streams N > 1 spreads the 32-layer workload's layers over N streams;
    any other workload, or N < 1, is refused before the GPU is touched."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode != 0
    assert "--streams N > 1 applies to --workload c3 only" in (r.stderr + r.stdout)
