"""The N-GPU bench is N independent replicas (the batch rows are independent, no
data-path collective): its host logic — barrier, the maximum of the per-rank
times, one distinct workload seed per rank, rank 0 alone running the reference
arm — checked with two gloo ranks on the CPU."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(dist)
        mx = bench.max_over_ranks(10.0 * (rank + 1), dist)
        # the reference arm runs on rank 0 only: the others return without work
        skipped = bench.run_reference(None, world, rank, dist) is None if rank != 0 else True
        bench.barrier(dist)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{mx} {skipped}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max(tmp_path):
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        mx, skipped = open(tmp_path / f"rank{r}.txt").read().split()
        assert float(mx) == 20.0 and skipped == "True"


def test_replicas_draw_distinct_workloads():
    from hybrid_sparse_attention_gb300 import synth
    base = synth.SEED["c4layer"]
    a = synth.c4_lengths(base, 64)
    b = synth.c4_lengths(base + 1000, 64)   # rank 1's seed in bench.build_workload
    assert not torch.equal(a, b)
    assert torch.equal(a, synth.c4_lengths(base, 64))
