"""Multi-process path of bench.py on CPU (gloo, world size 2): the job's step
time is the slowest rank's and its token count the sum over ranks, so the
reported throughput is whole-job; each rank otherwise runs its own replica
(weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import sys
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    ms, tokens = bench.aggregate([1.25, 3.5][rank], [17, 40][rank], ws, "cpu")
    # (the end-to-end figure passes a mean number of tokens per step)
    _, frac = bench.aggregate(1.0, [2.5, 0.25][rank], ws, "cpu")
    dist.barrier()
    q.put((rank, ms, tokens, frac))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 3.5, 57, 2.75), (1, 3.5, 57, 2.75)]


def test_single_rank_is_untouched():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.aggregate(2.0, 9, 1, "cpu") == (2.0, 9)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm (the oracle on host cores) runs on
    rank 0 alone; another rank exits 0 at once and prints nothing."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
