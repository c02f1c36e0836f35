"""The bench's multi-rank host logic on CPU: two gloo ranks (world size 2), as
torchrun launches them.  Each rank runs its own replica of the step; the job's time
is the slowest rank's, and the value counts the work of every rank.  No GPU."""

import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    try:
        r, w = bench.dist_setup(None)
        bench.barrier(w)
        # rank 1 is the slower replica: 30 ms for its 5 steps against 20 ms
        ms_rank = 20.0 + 10.0 * r
        ms_max = bench.all_max(ms_rank, w)
        value = bench.replicas_value(ms_max, 5, 2.0 * 8192 ** 3, w)
        bench.barrier(w)
        dist.destroy_process_group()
        q.put((r, w, ms_max, value))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, -1, repr(e), None))


def test_two_gloo_ranks_agree_on_slowest_time_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2, 2], out
    assert [o[2] for o in out] == [30.0, 30.0]
    # 2 replicas x 5 steps x 2*8192^3 FLOP in 30 ms
    want = 2 * 5 * 2.0 * 8192 ** 3 / 0.030 / 1e12
    assert abs(out[0][3] - want) < 1e-9 * want and out[0][3] == out[1][3]


def test_one_rank_is_plain_single_process():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.all_max(12.5, 1) == 12.5
    assert bench.replicas_value(10.0, 4, 1e12, 1) == 400.0


def test_reference_arm_non_zero_rank_exits_quietly():
    # Under torchrun only rank 0 times the oracle; the other ranks exit 0 with no output.
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
