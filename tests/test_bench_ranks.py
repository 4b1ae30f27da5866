"""The benchmark's multi-rank host logic on the CPU: gloo ranks, no GPU.

`bench.py --gpus N` runs N independent replicas (one process per GPU) that
meet at a barrier around the timed region; the step time is the maximum
over ranks and only rank 0 prints.  These tests run that logic with two
gloo ranks, and the reference arm's rule that only rank 0 does work.
"""

import json
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


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    bench.barrier(world)
    got = bench.max_over_ranks(1.0 + 2.5 * rank, world)
    bench.barrier(world)
    out.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(out.get(timeout=5) for _ in procs)
    assert got == {0: 3.5, 1: 3.5}


def _bench_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                           "tiny", "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_runs_on_rank_zero_only():
    other = _bench_reference(1, 2)
    assert other.returncode == 0 and other.stdout.strip() == ""
    first = _bench_reference(0, 2)
    assert first.returncode == 0, first.stderr[-2000:]
    lines = [l for l in first.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
