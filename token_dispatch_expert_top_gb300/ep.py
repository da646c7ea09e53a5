"""Expert-parallel plan of the MoE layer across R ranks: host-side index bookkeeping.

The pages' layer runs expert parallel ([MoK-2.37x] = "Cursor's MoK achieves 2.37x
performance boost on NVIDIA GB300 NVL72", section 01: the experts are split across
GPUs and every token stays on its data-parallel rank, so the forward exchanges
tokens once each way; section 02: the expert rank pulls the rows its schedule
lists from the source ranks' memory, and the expert outputs are pushed back to
the tokens' ranks).  On one GPU the same schedule runs over virtual shards in
local HBM; this module says which part of that schedule each rank of an R-way
expert-parallel layer owns, and how the pushed rows are addressed.  It holds no
step of the layer's arithmetic.

Conventions (the single-GPU library's, cut R ways):
  * tokens: N = R * N_r, rank s holds tokens [s*N_r, (s+1)*N_r); each rank's
    block is S/R of the layer's S virtual shards, so shard c lives on rank
    c // (S/R) as its local shard c % (S/R);
  * experts: rank r owns the contiguous range expert_ranges(E, R)[r];
  * the layout (counts, offsets, sched, inv) is the single-GPU one over all N
    tokens -- each rank computes it from the all-gathered top-k indices --
    so slots are expert-major and ascending in token index inside an expert.
    Rank r's slots are then one contiguous range, [offsets[e_lo], offsets[e_hi]).
"""
from __future__ import annotations

import numpy as np


def expert_ranges(E: int, R: int) -> list[tuple[int, int]]:
    """Contiguous expert ranges of R ranks, sizes differing by at most one (the
    first E % R ranks hold one more)."""
    if R < 1 or E < R:
        raise ValueError(f"cannot split {E} experts over {R} ranks")
    base, extra = divmod(E, R)
    out, lo = [], 0
    for r in range(R):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def expert_owner(E: int, R: int) -> np.ndarray:
    """owner[e] = the rank that holds expert e."""
    owner = np.empty(E, dtype=np.int32)
    for r, (lo, hi) in enumerate(expert_ranges(E, R)):
        owner[lo:hi] = r
    return owner


def slot_range(offsets: np.ndarray, E: int, R: int, r: int) -> tuple[int, int]:
    """(first slot, slot count) of rank r's experts in the global layout."""
    lo, hi = expert_ranges(E, R)[r]
    return int(offsets[lo]), int(offsets[hi] - offsets[lo])


def pull_schedule(sched: np.ndarray, offsets: np.ndarray, E: int, R: int, S: int, r: int) -> np.ndarray:
    """Rank r's pull schedule: for each of its slots in slot order, (source rank,
    source-local shard, row) -- the (shard, row) pairs of the global schedule with
    the shard resolved to the rank whose memory holds it."""
    if S % R:
        raise ValueError(f"{S} shards do not split over {R} ranks")
    first, count = slot_range(offsets, E, R, r)
    sr = np.asarray(sched[first:first + count], dtype=np.int64)
    per = S // R
    return np.stack([sr[:, 0] // per, sr[:, 0] % per, sr[:, 1]], axis=1).astype(np.int32)


def push_plan(inv: np.ndarray, idx: np.ndarray, offsets: np.ndarray, E: int, R: int, N: int):
    """How the expert outputs go back to the tokens' ranks.

    Returns (dest, send) where
      dest[n, j] = (expert rank, slot within that rank's range) of choice j of
                   token n: where token n's rank finds that choice's y row among
                   the rows the expert rank pushed;
      send[r][s] = the local slots (ascending) whose y rows expert rank r pushes
                   to source rank s, in the order it sends them.
    """
    N_r = N // R
    owner = expert_owner(E, R)
    ranges = [slot_range(offsets, E, R, r) for r in range(R)]
    first = np.array([f for f, _ in ranges], dtype=np.int64)
    e_of = owner[np.asarray(idx, dtype=np.int64)]
    dest = np.stack([e_of, np.asarray(inv, dtype=np.int64) - first[e_of]], axis=-1).astype(np.int32)
    send = [[None] * R for _ in range(R)]
    tok_rank = np.arange(N) // N_r
    for r in range(R):
        for s in range(R):
            mine = (e_of == r) & (tok_rank[:, None] == s)
            send[r][s] = np.sort(dest[..., 1][mine]).astype(np.int64)
    return dest, send


def receive_index(dest: np.ndarray, send, s: int, N: int, R: int) -> np.ndarray:
    """For source rank s: position of each (local token, choice) y row in the
    concatenation, over expert ranks r = 0..R-1, of the rows r pushed to s (each in
    send[r][s] order).  Returns an [N_r, k] index into that concatenation."""
    N_r = N // R
    mine = dest[s * N_r:(s + 1) * N_r]
    base = 0
    pos = np.empty(mine.shape[:2], dtype=np.int64)
    for r in range(R):
        lst = send[r][s]
        at = {int(v): i for i, v in enumerate(lst)}
        for n, j in zip(*np.nonzero(mine[..., 0] == r)):
            pos[n, j] = base + at[int(mine[n, j, 1])]
        base += len(lst)
    return pos
