"""Body of one rank for test_bench_ranks.py (a module of its own so that spawned
processes can import it)."""
import argparse
import os
import sys

import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        # each rank's own timed region; rank r is slower by 5 ms per rank
        t_ms = bench.max_over_ranks(100.0 + 5.0 * rank, world)
        rate = bench.job_rate(8192, 20, t_ms, world)
        args = argparse.Namespace(workload="tiny_f32", sample_tokens=2, steps=1, warmup=3)
        ref = bench.reference_arm(args, rank, world) if rank != 0 else "rank0"
        dist.barrier()
        q.put((rank, t_ms, rate, ref))
    finally:
        dist.destroy_process_group()
