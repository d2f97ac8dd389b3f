"""The multi-GPU form of the benchmark is independent replicas (every (b, h)
slice is independent, so nothing is exchanged on the data path); its only
cross-rank steps are the reductions of the timing (max of the ranks' times)
and of the units (sum).  Checked here with world_size 2 on the gloo backend,
CPU only."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        t_max = bench.reduce_replicas(1.5 + rank, "max")       # each rank's time
        units = bench.reduce_replicas(10.0 * (rank + 1), "sum")  # each rank's FLOPs
        q.put((rank, t_max, units))
    finally:
        dist.destroy_process_group()


def test_replica_reductions_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.reduce_replicas(3.25, "max") == 3.25
    assert bench.reduce_replicas(7.0, "sum") == 7.0


def test_reference_arm_under_torchrun_prints_once():
    """--impl reference under a 2-rank launch: rank 0 alone times the oracle
    and prints one JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
