"""The N > 1 host logic of bench.py, on CPU with two gloo ranks.

The layer shards over (sequence, head) with no collective, so the only
multi-rank code is the benchmark's: rank discovery from the launcher's
environment, the process group, the barriers around the timed region and the
max over ranks of the timings.  Each rank here runs in its own spawned
process with no GPU visible, so the group is gloo.
"""
import importlib.util
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    b = _bench()
    r, w, local = b.dist_info()
    dist = b.init_dist(w, local)
    b.barrier(dist)
    # each rank reports its own time; every rank must see the slowest
    m = b.max_over_ranks(dist, 10.0 + 5.0 * rank)
    b.barrier(dist)
    q.put((r, w, dist.get_backend(), m))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, "gloo", 15.0), (1, 2, "gloo", 15.0)]


def test_single_rank_needs_no_group():
    b = _bench()
    assert b.init_dist(1, 0) is None
    assert b.max_over_ranks(None, 3.5) == 3.5
    b.barrier(None)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "", "a rank other than 0 must print nothing"
