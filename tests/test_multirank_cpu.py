"""The N > 1 path of bench.py on CPU: two ranks over gloo (127.0.0.1).

The decode path shards by independent rows and requests, so the bench runs N
independent replicas; what the ranks share is the timing protocol: a barrier
on both sides of the timed region, the maximum of the per-rank step times,
and rank 0 alone printing the line.  These tests run that protocol (the
bench's own helpers) in two spawned processes."""
import json
import os
import socket
import subprocess
import sys

import multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    w, r, local, pg = bench.dist_setup()
    dev = torch.device("cpu")
    bench.barrier(pg, dev)
    ms_max = bench.reduce_max(pg, times[rank], dev)
    bench.barrier(pg, dev)
    out.put({"rank": r, "world": w, "local": local, "ms_max": ms_max,
             "value": bench.aggregate_value(w, 1000.0, ms_max)})
    pg.destroy_process_group()


def test_two_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    times = [3.5, 7.25]  # per-rank ms per step
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((out.get(timeout=180) for _ in procs), key=lambda d: d["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [d["rank"] for d in res] == [0, 1]
    assert all(d["world"] == 2 and d["ms_max"] == 7.25 for d in res)
    # weak scaling: both ranks' units over the slowest rank's time
    assert all(abs(d["value"] - 2 * 1000.0 / 7.25e-3) < 1e-6 for d in res)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "0"],
                          env=env, capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr[-2000:]
    assert proc.stdout.strip() == ""


def test_aggregate_value_is_whole_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_value(1, 8.0e6, 2.0) == 8.0e6 / 2.0e-3
    assert bench.aggregate_value(4, 8.0e6, 2.0) == 4 * 8.0e6 / 2.0e-3
    json.dumps({"value": bench.aggregate_value(2, 1.0, 1.0)})
