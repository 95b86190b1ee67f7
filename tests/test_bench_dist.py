"""bench.py's multi-rank host logic on CPU with gloo, world size 2: the
max-over-ranks step time, the sum of the ranks' work, the per-rank workload seeds, and a torchrun launch
of the reference arm (rank 0 alone prints one JSON line, the other rank exits
0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    m = bench.dist_max(1.5 + rank, world)
    total = bench.dist_sum(10.0 + rank, world)
    bench.barrier(world)
    spec = bench.rank_spec(workloads.config("tiny_bf16"), rank)
    out.put((rank, m, spec.seed, total))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_dist_helpers_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _, _ in res] == [2.5, 2.5]       # the max over ranks, seen by both
    assert res[0][2] != res[1][2]                          # each rank draws its own batch
    assert [t for _, _, _, t in res] == [21.0, 21.0]       # work summed over ranks


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-side launch test (no GPU use)")
def test_torchrun_reference_arm_world_2():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny_bf16"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
