"""The multi-GPU bench path on CPU: world-size-2 gloo ranks check the max-over-ranks timing
reduction and that only rank 0 runs (and prints) the reference arm."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max([1.0 + rank, 10.0 - rank, 0.5 * rank])
        assert bench.dist_env() == (rank, world, rank)

        class A:
            steps, warmup = 1, 3
        ref = bench.run_reference(A, rank, world) if rank != 0 else "skipped"
        out.put((rank, got, ref))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.timeout(120)
def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    (r0, got0, _), (r1, got1, ref1) = res
    assert got0 == got1 == [2.0, 10.0, 0.5]
    assert ref1 is None              # the reference arm runs on rank 0 only


@pytest.mark.timeout(300)
def test_gpus_flag_starts_the_ranks_itself():
    """`bench.py --gpus 2` with no external launcher starts two ranks (gloo on CPU for the
    reference arm); rank 0 alone prints one JSON line that reports both ranks."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                          "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--ref-budget-s", "1"], env=env, capture_output=True, text=True,
                         timeout=280)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
