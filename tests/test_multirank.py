"""The N>1 bench path on CPU: world_size-2 gloo ranks, each timing its own
replica; the job's time is the slowest rank and the value counts all ranks'
work (replicas only: no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = 10.0 + 5.0 * rank  # rank 1 is slower
    slow = bench.max_over_ranks(local_ms)
    rate = bench.whole_job_rate(1.0e9, world, slow)
    q.put((rank, slow, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_and_sum_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] == pytest.approx(2 * 1.0e9 / 0.015)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(2.0, 1, 1000.0) == 2.0


def test_bench_spawns_replica_ranks_itself():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (through
    torch.distributed.run); with the CPU stand-in step they use gloo, each picks the
    device of its local rank, and rank 0 reports the slowest rank's time and the
    work of both."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                            "MASTER_PORT")}
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--stub-step", "--steps", "5",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300, cwd=root)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout  # rank 0 alone prints
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["stub"] is True
    assert rec["devices"] == ["cpu:0", "cpu:1"]
    assert rec["ms_per_step"] == pytest.approx(max(rec["per_rank_ms"]))
    # rank 1's stand-in step sleeps 4 ms, rank 0's 2 ms: the job runs at the slower rank's pace
    assert rec["ms_per_step"] >= 4.0
    assert rec["value"] == pytest.approx(2 * 1.0 / (rec["ms_per_step"] * 1e-3))
