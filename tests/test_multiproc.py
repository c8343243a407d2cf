"""Multi-process host logic of the benchmark's replica mode, on CPU with the
gloo backend at world size 2: rendezvous on 127.0.0.1, barrier, the
max-over-ranks timing reduction, and the reference arm's rank-0-only rule
(other ranks exit without work)."""

import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_init(None)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 * (r + 1), w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, m))


def test_replicas_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 20.0), (1, 2, 20.0)]


def test_reference_arm_nonzero_rank_exits_quietly():
    """Under torchrun the reference arm runs on rank 0 only; rank 1 returns
    without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="1", LOCAL_RANK="0")
    code = ("import sys; sys.path.insert(0, %r); import bench; "
            "print(bench.run_reference(type('A', (), {'steps': 1, 'warmup': 3})(), 2, 1))" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "None"
