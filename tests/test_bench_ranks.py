"""bench.py's multi-rank rules on two gloo ranks (CPU processes): the timed figure
is the slowest rank's, `value` counts the units of every rank (replicas: each rank
runs the whole layer on its own GPU), and the reference arm does its work on rank 0
only."""
import multiprocessing as mp
import socket

import rank_worker


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_max_time_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=rank_worker.run, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, t_ms, rate, ref = q.get(timeout=120)
        res[r] = (t_ms, rate, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 105.0          # max over ranks
    assert res[0][1] == res[1][1] == 2 * 8192 * 20 / 0.105
    assert res[1][2] is None                          # reference arm: no work off rank 0
