"""Multi-process host logic on the CPU (gloo, world size 2, 127.0.0.1).

The operator runs as independent replicas, one per GPU, with no exchange step; what N > 1
adds is the bench's rank setup, the barrier around the timed region and the maximum of the
timings over ranks.  These run here as two gloo ranks, and `bench.py --impl reference` is
launched the way the driver launches it (torch.distributed.run, two ranks): rank 0 alone prints
the line, rank 1 exits 0 without work.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(world)]
    bench = _load_bench()
    args = bench.parse()
    w, r = bench.dist_setup(args)
    bench.barrier(w)
    # each rank reports its own time; every rank must see the maximum
    mx = bench.max_over_ranks(10.0 + 5.0 * r, w)
    bench.barrier(w)
    import torch.distributed as dist
    out.put((r, w, mx, dist.get_backend()))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[2] == 15.0 and g[3] == "gloo" for g in got)


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1",
           "--workload", "tiny_L2048"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
