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


def test_bench_gpus_2_self_launches_two_replicas():
    """`bench.py --gpus 2` without a torchrun environment re-launches itself
    with two ranks; rank 0 prints one line whose latency is the slower rank's
    (not divided by the rank count) and whose aggregate throughput counts both
    replicas."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["OMP_NUM_THREADS"] = "1"
    script = os.path.join(ROOT, "tests", "replica_stub_bench.py")
    r = subprocess.run([sys.executable, script, "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2
    assert abs(line["value"] - 110.0) < 1e-6            # max over ranks, in us
    assert abs(line["e2e"]["value"] - 220.0) < 1e-6
    assert abs(line["throughput_all_replicas"]["value"] - 2 * 64 / 110e-6) < 1e-3
    assert line["config"]["parallelism"] == "replicas x2"


def test_bench_rejects_mismatched_world_size():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    script = os.path.join(ROOT, "tests", "replica_stub_bench.py")
    r = subprocess.run([sys.executable, script, "--gpus", "2"], capture_output=True, text=True,
                       env=env, timeout=120)
    assert r.returncode != 0 and "--gpus 2" in (r.stderr + r.stdout)
