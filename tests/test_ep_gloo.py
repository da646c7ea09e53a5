"""The forward layer split expert parallel over two gloo ranks (CPU processes):
each rank routes its own tokens, the top-k indices are all-gathered, each rank
pulls the rows of its experts' slots by its pull schedule from a per-rank table
of source rows, runs its experts on the oracle, and pushes every output row back
to its token's rank, which combines.  The union of the ranks' outputs must equal
the oracle's single-process forward."""
import multiprocessing as mp
import socket

import numpy as np
import pytest

import ep_worker
from token_dispatch_expert_top_gb300 import ep


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_expert_ranges_cover_every_expert_once():
    for E, R in ((8, 2), (7, 3), (256, 8), (5, 5)):
        rg = ep.expert_ranges(E, R)
        assert rg[0][0] == 0 and rg[-1][1] == E
        assert all(a[1] == b[0] for a, b in zip(rg, rg[1:]))
        sizes = [hi - lo for lo, hi in rg]
        assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        ep.expert_ranges(2, 3)


def test_push_plan_is_a_bijection():
    rng = np.random.default_rng(0)
    N, k, E, R, S = 48, 3, 6, 3, 6
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(N)]).astype(np.int32)
    # a stable counting layout, expert-major (the single-GPU layout)
    order = np.argsort(idx.ravel(), kind="stable")
    inv = np.empty(N * k, dtype=np.int64)
    inv[order] = np.arange(N * k)
    inv = inv.reshape(N, k)
    offsets = np.concatenate([[0], np.cumsum(np.bincount(idx.ravel(), minlength=E))])
    dest, send = ep.push_plan(inv, idx, offsets, E, R, N)
    seen = set()
    for r in range(R):
        first, cnt = ep.slot_range(offsets, E, R, r)
        slots = np.concatenate([send[r][s] for s in range(R)])
        assert sorted(slots.tolist()) == list(range(cnt))         # every slot pushed exactly once
        for s in range(R):
            pos = ep.receive_index(dest, send, s, N, R)
            assert pos.shape == (N // R, k)
        seen.update((r, int(v)) for v in slots)
    assert len(seen) == N * k


@pytest.mark.parametrize("wk", [
    dict(name="ep_bf16", N=96, H=64, I=64, E=8, k=2, S=4, dtype="bf16"),
    dict(name="ep_mxfp8_skew", N=128, H=64, I=64, E=6, k=3, S=4, dtype="mxfp8", skew=1.0),
], ids=lambda d: d["name"])
def test_two_gloo_ranks_expert_parallel_forward_equals_oracle(wk):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=ep_worker.run, args=(r, 2, port, q, wk)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, v = q.get(timeout=180)
        assert not isinstance(v, str), v
        res[r] = v
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    idx_same, max_diff, n_diff, pulls = res[0]
    assert idx_same
    assert sum(pulls) == wk["N"] * wk["k"] and min(pulls) > 0
    assert n_diff == 0 and max_diff == 0.0, (max_diff, n_diff)
