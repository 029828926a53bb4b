"""The multi-rank path of bench.py on CPU: two gloo ranks, launched as
processes the way torchrun launches the GPU ranks (one process per rank,
rendezvous on 127.0.0.1). The bench runs one replica of the workload per rank
(rows are independent: no collective on the data path); the only collectives
are the barrier around the timed region and the max over ranks of the time."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws_env, rank_env, local = bench.dist_info()
    bench.maybe_init_dist(ws_env, "gloo")
    bench.barrier(ws_env)
    # rank r takes 2 + r ms per step over 1000 units
    value, ms = bench.job_throughput(1000, 2.0 + rank_env, ws_env, "cpu")
    q.put((rank_env, local, value, ms))
    bench.barrier(ws_env)
    torch.distributed.destroy_process_group()


def test_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and [o[1] for o in out] == [0, 1]
    for _, _, value, ms in out:
        assert ms == 3.0                          # the slowest rank's time
        assert value == pytest.approx(2 * 1000 / 3e-3)


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(500, 4.0, 1, "cpu")
    assert ms == 4.0 and value == pytest.approx(500 / 4e-3)


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched by torchrun with 2 ranks: rank 0 alone
    prints one JSON line (the oracle timed on the host), the other rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
