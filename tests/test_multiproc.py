"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2).

The decode path has no exchange step, so more GPUs mean independent
replicas: each rank times its own replica, rank 0 prints the one JSON line,
and the step time is the maximum over ranks.  These tests run that host
logic as two processes on the CPU -- the helpers directly, and the whole
reference arm launched as a multi-GPU run launches bench.py (torch.distributed.run)."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup()
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + 5.0 * r, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((r, w, local, got))


def test_bench_helpers_on_two_gloo_ranks():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0, p.exitcode
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, *_ in res] == [0, 1]
    assert all(w == world for _, w, _, _ in res)
    assert [loc for _, _, loc, _ in res] == [0, 1]
    assert all(got == 15.0 for *_, got in res)  # the maximum over ranks, on every rank


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "1", "--ref-step-s", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
