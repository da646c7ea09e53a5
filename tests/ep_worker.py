"""Body of one rank for test_ep_gloo.py (a module of its own so that spawned
processes can import it): the forward layer expert parallel over gloo ranks,
each rank's compute done by the oracle."""
import os
import sys

import numpy as np
import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(rank: int, world: int, port: int, q, wk: dict) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for p in (ROOT, os.path.join(ROOT, "oracle")):
            sys.path.insert(0, p)
        import oracle as O
        from token_dispatch_expert_top_gb300 import ep, synth

        w = synth.Workload(**wk)
        N, H, E, k, S = w.N, w.H, w.E, w.k, w.S
        inp = synth.make_inputs(w, device="cpu")       # every rank draws the same seeded layer
        N_r = N // world
        mine = slice(rank * N_r, (rank + 1) * N_r)
        x = O._f64(inp["x"])

        # 1. each rank routes its own tokens; the top-k indices are all-gathered
        logits = O.router_logits(x[mine], inp["w_router"], inp["bias"])
        idx_l, gate_l = O.route_topk(logits, k)
        parts = [torch.empty((N_r, k), dtype=torch.int32) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(idx_l))
        idx = torch.cat(parts).numpy()
        counts, offsets, sched, inv = O.layout(idx, E, S)

        # 2. the source ranks' rows (quantised at the source for MXFP8), reached
        #    through a table with one entry per rank (peer memory, emulated)
        src = O.mxfp8_values(x[mine]) if O.FORMATS[w.dtype][0] == "mxfp8" else x[mine]
        table = [torch.empty((N_r, H), dtype=torch.float64) for _ in range(world)]
        dist.all_gather(table, torch.from_numpy(np.ascontiguousarray(src)))
        table = [t.numpy() for t in table]

        # 3. pull this rank's slots by its schedule; expert FFN of its experts
        ps = ep.pull_schedule(sched, offsets, E, world, S, rank)
        rows = N // S
        first, cnt = ep.slot_range(offsets, E, world, rank)
        a = np.zeros((cnt, H))
        for i, (s, ls, r) in enumerate(ps):
            a[i] = table[s][ls * rows + r]
        y = np.zeros((cnt, H))
        e_lo, e_hi = ep.expert_ranges(E, world)[rank]
        for e in range(e_lo, e_hi):
            lo, hi = offsets[e] - first, offsets[e + 1] - first
            if hi > lo:
                wg, wu, wd = O.expert_operands(inp["w_gate_up"][e], inp["w_down"][e], w.dtype)
                y[lo:hi] = O.expert_ffn(a[lo:hi], wg, wu, wd, w.dtype)

        # 4. push every y row to its token's rank (point to point), combine there
        dest, send = ep.push_plan(inv, idx, offsets, E, world, N)
        reqs, got = [], []
        for s in range(world):
            if s != rank:
                reqs.append(dist.isend(torch.from_numpy(np.ascontiguousarray(y[send[rank][s]])), s))
        for r in range(world):
            if r == rank:
                got.append(y[send[rank][rank]])
            else:
                buf = torch.empty((len(send[r][rank]), H), dtype=torch.float64)
                dist.recv(buf, r)
                got.append(buf.numpy())
        for rq in reqs:
            rq.wait()
        ycat = np.concatenate(got) if got else np.zeros((0, H))
        pos = ep.receive_index(dest, send, rank, N, world).astype(np.int32)
        out = O.round_to(O.combine(ycat, pos, gate_l), O.FORMATS[w.dtype][3])

        outs = [torch.empty((N_r, H), dtype=torch.float64) for _ in range(world)]
        dist.all_gather(outs, torch.from_numpy(np.ascontiguousarray(out)))
        res = None
        if rank == 0:
            ref = O.forward(inp, E, k, S, w.dtype)
            got_out = torch.cat(outs).numpy()
            res = (bool(np.array_equal(idx, ref["idx"])),
                   float(np.abs(got_out - ref["out"]).max()),
                   int(np.count_nonzero(got_out != ref["out"])),
                   [len(ep.pull_schedule(sched, offsets, E, world, S, r)) for r in range(world)])
        q.put((rank, res))
    except Exception as exc:          # report instead of leaving the parent waiting
        q.put((rank, f"error: {type(exc).__name__}: {exc}"))
        raise
    finally:
        dist.destroy_process_group()
