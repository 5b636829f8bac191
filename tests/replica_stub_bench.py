"""Entry script for tests/test_replicas.py: bench.py's own launch path
(self-relaunch under torch.distributed.run, rendezvous, barrier, maximum over
ranks, one line from rank 0) with the per-rank GPU measurement replaced by a
CPU stub whose per-rank times are known."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def stub_measure(args, rank, local, dist):
    bench.barrier(dist)
    ms = 0.100 + 0.010 * rank          # rank r: (100 + 10 r) us per layer
    line = bench.base_line(args, 1, bench.METRIC, "us", False, bench.WORKLOAD, ms * 1000)
    line["e2e"] = {"value": None, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    line["rank_seed"] = bench.synth.SEED["c4layer"] + 1000 * rank
    bench.barrier(dist)
    return {"ms": ms, "e2e_ms": 2 * ms, "line": line, "units_per_step": 1,
            "tokens_per_step": 64, "throughput_unit": "decode tokens/s through one layer"}


if __name__ == "__main__":
    bench.main(measure=stub_measure)
