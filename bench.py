#!/usr/bin/env python3
"""Benchmark of the decode-time hybrid sparse-attention hot path.

One step = one decode step of one C4 hybrid layer through the C ABI
(hsa_layer_decode): append the new token, compress the completed 4-token
blocks, score every C4 entry with the indexer, select the top-512, and attend
the 128-token window plus the selected entries.  Workload: batch 64, context
lengths uniform in [16,384, 131,072], 64 query heads of 512 latent + 64 rope
channels sharing one KV head, indexer 8 heads x 128, window 128, top-512,
bf16 storage, fp32 accumulation, synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hsa|reference]
                    [--config c4layer|topk|compress|longctx]

Prints one JSON line (rank 0).  With --gpus N > 1 (and no torchrun
environment) the script re-launches itself under torch.distributed.run with N
ranks; every rank runs an independent replica of the workload (its own seed):
weak scaling, no data-path collective.  The reported latency is the maximum
over ranks; the aggregate throughput of all replicas is a separate key.

--config picks the headline line: the C4 layer (default; its line also carries
the other configurations' timings as extra keys), the standalone top-k
(64 x 262,144), the standalone compressor (32 x 65,536 x 512 at r = 4 and 128)
or the 1M-token pair (C4 and C128 layers, batch 4).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hybrid_sparse_attention_gb300 import _lib, synth  # noqa: E402

METRIC = "us per decode layer (C4+SWA, 128K ctx, batch 64)"
WORKLOAD = ("C4 hybrid decode layer: B=64, L~U[16384,131072], Hq=64, Dqk=576 (512+64), Dv=512, "
            "indexer Hi=8 Di=128, top-k 512, SWA window 128, 1 query token")
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def layer_bytes(L, shape, kind=4, key_entry_bytes=None, T=1):
    """Algorithmic HBM bytes of one layer step (each byte the method must move,
    counted once).  C4: indexer keys, score write + read, the gathered window
    and top-k rows, q, o, the index list, the new-token append and the 4-row
    block reads / writes of the sequences whose block completes.  C128: the
    gathered window and every C128 row, q, o, the append and the 128-row
    block compression of the sequences whose block completes.
    key_entry_bytes: bytes of one stored indexer key (bf16: 2 Di; E4M3 codes
    and their fp32 scale: Di + 4).  T query tokens per step (L: tokens after
    it): the keys are read once for all tokens; scores, gathers, q, o, the
    index lists and the appended rows count once per token."""
    L = L.to(torch.int64)
    B = L.numel()
    D, Di = shape.Dqk, shape.Di
    Lt = [L - (T - 1 - t) for t in range(T)]   # each token's length
    win = sum(int(torch.clamp(x, max=shape.W).sum()) for x in Lt)
    q = T * B * shape.Hq * D * 2
    o = T * (B * shape.Hq * shape.Dv * 2 + B * shape.Hq * 4)
    if kind == 128:
        n = L // 128
        gather = (win + int(n.sum())) * D * 2
        append = B * (D * 2 * 2 + D * 2 * 3)              # read kv, z rows; write window + rings
        ncomp = int((L % 128 == 0).sum())
        compress = ncomp * (128 * 2 * D * 2 + D * 2)
        total = gather + q + o + append + compress
        return {"total": total, "gather": gather, "attention": gather + q + o,
                "append_compress": append + compress}
    n4 = L // 4
    N = int(n4.sum())
    Nt = sum(int((x // 4).sum()) for x in Lt)            # scores over all tokens
    kb = Di * 2 if key_entry_bytes is None else key_entry_bytes
    keys = N * kb
    iq_w = T * B * shape.Hi * (Di * 2 + 4)
    scores = 2 * Nt * 4
    gather = (win + sum(int(torch.clamp(x // 4, max=shape.k).sum()) for x in Lt)) * D * 2
    idx = 2 * T * B * shape.k * 4
    append = T * B * (D * 2 * 2 + D * 2 * 3 + Di * 2 * 2 + Di * 2 * 2)   # read new rows, write rings
    ncomp = int(((L // 4) != ((L - T) // 4)).sum())
    compress = ncomp * (4 * 2 * (D + Di) * 2 + D * 2 + kb)
    indexer = keys + iq_w + Nt * 4
    total = keys + iq_w + scores + gather + q + o + idx + append + compress
    return {"total": total, "indexer": indexer, "keys": keys, "gather": gather,
            "attention": gather + q + o + idx // 2, "topk": Nt * 4 + idx // 2,
            "append_compress": append + compress}


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def relaunch(n, argv):
    """Runs this script again under torch.distributed.run with n local ranks
    (rendezvous on 127.0.0.1); returns its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.abspath(sys.argv[0])] + list(argv)
    return subprocess.call(cmd)


def dist_setup(gpu=True):
    """(world, rank, local rank, torch.distributed or None) from the torchrun
    environment; NCCL between GPU ranks, gloo when the measurement is a CPU stub."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if gpu:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
        return world, rank, local, dist
    return 1, 0, local, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle arm

def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def sample_state(g, seqs):
    """numpy copy (oracle input) of sequences `seqs` of a layer state."""
    offs = g.pool_offsets.cpu()
    c4 = g.kind == 4
    kv = torch.cat([g.kv_pool[int(offs[b]):int(offs[b + 1])] for b in seqs])
    caps = torch.tensor([int(offs[b + 1] - offs[b]) for b in seqs], dtype=torch.int64)
    new_offs = torch.zeros(len(seqs) + 1, dtype=torch.int64)
    new_offs[1:] = torch.cumsum(caps, 0)
    sel = torch.tensor(seqs, device=g.q.device)
    s = {"kind": g.kind, "ratio": g.ratio, "Dv": g.shape.Dv, "k": g.shape.k if c4 else 0,
         "scale": g.shape.scale, "pool_offsets": new_offs.numpy(),
         "seq_len_in": g.seq_len_in[sel].cpu().numpy(), "kv_pool": _bits(kv),
         "b_kv": g.b_kv.cpu().numpy()}
    names = ["swa", "kv_ring", "z_ring", "kv_new", "z_new", "q"]
    if c4:
        key = torch.cat([g.key_pool[int(offs[b]):int(offs[b + 1])] for b in seqs])
        s.update(key_pool=_bits(key), b_ik=g.b_ik.cpu().numpy(), w=g.w[sel].cpu().numpy())
        names += ["ik_ring", "iz_ring", "ik_new", "iz_new", "iq"]
    for name in names:
        s[name] = _bits(getattr(g, name)[sel])
    return s


def oracle_threads():
    import oracle
    oracle.build()
    return oracle.hardware_threads()


def oracle_layer_runner(g):
    """One oracle decode step over the whole batch of layer state g.  The step
    rewrites the same ring slots and pool rows with the same values each time
    (its input lengths are not advanced), so repeated calls time the same
    step.  Returns (run, description of the threads that do the work)."""
    import oracle
    threads = oracle_threads()
    B = g.seq_len_in.numel()
    s = sample_state(g, list(range(B)))

    def run():
        oracle.layer_decode(s, threads=threads)

    busy = {"attention": min(threads, B * g.shape.Hq), "topk": min(threads, B),
            "indexer": threads if g.kind == 4 else 0, "compress": 1}
    return run, threads, busy


def time_oracle(run, budget_s, min_calls=1):
    """Calls run() until budget_s of wall time is spent (at least min_calls);
    returns (mean seconds per call, calls)."""
    spent, n = 0.0, 0
    while n < min_calls or spent < budget_s:
        t0 = time.perf_counter()
        run()
        spent += time.perf_counter() - t0
        n += 1
    return spent / n, n


# ----------------------------------------------------------------------------- main

def parse_args(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="hsa", choices=["hsa", "reference"])
    ap.add_argument("--config", default="c4layer", choices=["c4layer", "topk", "compress", "longctx"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline (0: skip)")
    ap.add_argument("--layers", type=int, default=60,
                    help="layers in the CUDA-graph multi-layer step measurement (0: skip)")
    ap.add_argument("--no-extra", action="store_true",
                    help="c4layer: skip the other configurations' timings")
    ap.add_argument("--profile", action="store_true",
                    help="profiling run, for ncu: build the workload of --config, run it twice "
                         "(c4layer: two layer steps; topk: two calls; compress: two calls at each "
                         "ratio on 4 sequences), exit")
    ap.add_argument("--profile-ctx", type=int, nargs=2, default=None, metavar=("LO", "HI"),
                    help="with --profile: context lengths ~ U[LO, HI] instead of the bench's "
                         "(a smaller case of the same layer for multi-pass ncu captures)")
    return ap.parse_args(argv)


def main(argv=None, measure=None):
    """measure: the per-rank measurement (default: the GPU measurement of
    --config); the replica logic around it is the same for any measurement."""
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch(args.gpus, argv))
    world, rank, local, dist = dist_setup(gpu=measure is None)
    try:
        if world != args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} but the launch has {world} ranks")
        if measure is None:
            torch.cuda.set_device(local)
        if args.impl == "reference":
            run_reference(args, world, rank, dist)
        elif args.profile:
            if args.config == "topk":
                run_profile_topk()
            elif args.config == "compress":
                run_profile_compress()
            else:
                run_profile(args.profile_ctx)
        else:
            run_hsa(args, world, rank, local, dist, measure)
    finally:
        if dist is not None:
            dist.destroy_process_group()


def build_workload(rank, ctx=None, device="cuda"):
    seed = synth.SEED["c4layer"] + 1000 * rank
    L = synth.c4_lengths(seed, 64) if ctx is None else synth.c4_lengths(seed, 64, ctx[0], ctx[1])
    g = synth.filled_state(seed, 4, synth.FULL, L, device=device)
    return L, g


def longctx_workload(kind, rank=0, device="cuda"):
    """The 1M-token pair: batch 4 at L = 1,048,576 tokens after this step (the
    step completes both a 4- and a 128-token block), the bench's head shapes."""
    seed = synth.SEED["longctx"] + 1000 * rank
    L = torch.full((4,), 1 << 20, dtype=torch.int32)
    g = synth.filled_state(seed, kind, synth.FULL, L, device=device, name=f"long{kind}")
    return L, g


def base_line(args, world, metric, unit, higher, workload, value):
    return {"metric": metric, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
            "higher_is_better": higher, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload, "parallelism": f"replicas x{world}"}}


def run_reference(args, world, rank, dist):
    """The oracle (plain CPU C++), as it stands, on the host cores, timed on
    the configuration's own workload: each step is one whole oracle step (the
    full 64-sequence layer for the default configuration).  Under torchrun
    only rank 0 runs it; the other ranks return without work."""
    if rank != 0:
        return None
    cfg = args.config
    if cfg == "c4layer":
        L, g = build_workload(0)
        run, threads, busy = oracle_layer_runner(g)
        metric, unit, workload, per = METRIC, "us", WORKLOAD, 1.0
        sample = "the whole 64-sequence layer step per timed step"
        to_value = lambda sec: sec * 1e6
        higher = False
    elif cfg == "longctx":
        L, g = longctx_workload(4)
        run, threads, busy = oracle_layer_runner(g)
        metric, unit, workload = LONG_METRIC, "us", LONG_WORKLOAD
        sample = "the whole batch-4 C4 layer step per timed step"
        to_value = lambda sec: sec * 1e6
        higher = False
    elif cfg == "topk":
        run, threads, busy, sample = oracle_topk_runner()
        metric, unit, workload = TOPK_METRIC, "rows/s", TOPK_WORKLOAD
        to_value = lambda sec: 64 / sec
        higher = True
    else:
        run, threads, busy, sample, scale = oracle_compress_runner(4)
        metric, unit, workload = COMPRESS_METRIC, "us", COMPRESS_WORKLOAD
        to_value = lambda sec: sec * scale * 1e6
        higher = False
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    v = to_value(sec)
    line = base_line(args, 1, metric, unit, higher, workload, v)
    line.update({"impl": "reference", "dtype": "f64", "ms_per_step": sec * 1000,
                 "cpu_baseline": {"value": v, "unit": unit, "cores": threads, "kind": "oracle",
                                  "sample": sample, "threads_busy_by_stage": busy},
                 "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0}})
    print(json.dumps(line), flush=True)
    return line


class L2Flush:
    """Evicts L2 between steps, outside the timed events: writes a buffer larger
    than L2, then reads another one, so that the lines left behind are clean and
    the next step does not pay for writing back the flush's own dirty data."""

    def __init__(self):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self, i):
        self.w.fill_(float(i))
        torch.sum(self.r, dim=0, out=self.sink)


L2_NOTE = (f"{L2_FLUSH_BYTES >> 20} MiB written, then {L2_FLUSH_BYTES >> 21} MiB read, before "
           "every step, outside the timed events (L2 cold and clean)")


def timed(fn, flush, warmup, steps, stream=None):
    """CUDA-event milliseconds of `steps` calls of fn() after `warmup` calls,
    L2 flushed before each, events on the launching stream."""
    stream = stream or torch.cuda.current_stream()
    for i in range(warmup):
        flush(i)
        fn()
    ts = []
    for i in range(steps):
        flush(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return ts


def run_hsa(args, world, rank, local, dist, measure=None):
    measure = measure or {"c4layer": measure_c4layer, "topk": measure_topk_line,
                          "compress": measure_compress_line,
                          "longctx": measure_longctx_line}[args.config]
    res = measure(args, rank, local, dist)
    # latency: the slowest replica; every replica runs the full workload
    ms_max = max_over_ranks(res["ms"], dist)
    e2e_max = max_over_ranks(res["e2e_ms"], dist) if res.get("e2e_ms") is not None else None
    if rank != 0:
        return None
    line = res["line"]
    higher = line["higher_is_better"]
    per_unit = res.get("units_per_step", 1)
    if higher:      # a rate: value is per replica-step units / time, summed over replicas
        line["value"] = world * per_unit / (ms_max * 1e-3)
    else:
        line["value"] = ms_max * 1000
    line["n_gpus"] = world
    line["ms_per_step"] = ms_max
    line["config"]["parallelism"] = f"replicas x{world}"
    line["throughput_all_replicas"] = {
        "value": world * res.get("tokens_per_step", per_unit) / (ms_max * 1e-3),
        "unit": res.get("throughput_unit", "units/s"),
        "note": "aggregate of every replica: each runs the full workload"}
    if e2e_max is not None:
        e = line["e2e"]
        e["value"] = world * per_unit / (e2e_max * 1e-3) if higher else e2e_max * 1000
    print(json.dumps(line), flush=True)
    return line


def layer_outputs(g):
    B, shape = g.seq_len_in.numel(), g.shape
    out = torch.empty(B, shape.Hq, shape.Dv, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, shape.Hq, dtype=torch.float32, device="cuda")
    seq_out = torch.empty_like(g.seq_len_in)
    idx = scores = None
    if g.kind == 4:
        idx = torch.empty(B, shape.k, dtype=torch.int32, device="cuda")
        scores = torch.empty(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
    return out, lse, seq_out, idx, scores


def rotating_us(steps_fns, warmup, steps, stream):
    """Mean CUDA-event microseconds of one step, step i running steps_fns[i mod
    n] (each on its own layer state: inputs larger than L2, no flush)."""
    n = len(steps_fns)
    for i in range(max(warmup, n)):
        steps_fns[i % n]()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        ev0[i].record(stream)
        steps_fns[i % n]()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in zip(ev0, ev1)) * 1000


def layer_variants(args, runs, peak):
    """The headline step in two variants, each over the same rotating layer
    states: (1) the top-k as its own kernels after the indexer instead of
    fused into the attention kernel (no overlap of the window's attention
    with the selection); (2) an E4M3 indexer-key pool (the states' bf16 key
    pools quantized per row by the library: codes plus one fp32 scale per
    entry; every other tensor as in the headline)."""
    import copy as _copy
    stream = torch.cuda.current_stream()
    out = {}
    # (1) separate top-k: a bound on the rows above the fused selection's limit
    descs = [_lib.layer_desc(r.g, r.out, r.lse, r.seq_out, None, r.scores, max_pool_rows=40000)
             for r in runs]
    wss = [_lib.workspace(_lib.hsa_layer_decode_workspace_size(d)) for d in descs]
    us = rotating_us([lambda d=d, w=w: _lib.hsa_layer_decode(d, ws=w) for d, w in zip(descs, wss)],
                     args.warmup, args.steps, stream)
    out["topk_separate_kernels"] = {"us": us, "launches": _lib.hsa_layer_decode_launches(descs[0])}
    del descs, wss
    # (2) E4M3 key pools
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in stage:
        e.record(stream)
    fns, stage_fns, keep = [], [], []
    for r in runs:
        g8 = _copy.copy(r.g)
        g8.key_pool, g8.key_scale = _lib.hsa_quantize_e4m3(r.g.key_pool.float())
        d = _lib.layer_desc(g8, r.out, r.lse, r.seq_out, None, r.scores)
        ds = _lib.layer_desc(g8, r.out, r.lse, r.seq_out, None, r.scores,
                             stage_events=[e.cuda_event for e in stage])
        w = _lib.workspace(_lib.hsa_layer_decode_workspace_size(d))
        fns.append(lambda d=d, w=w: _lib.hsa_layer_decode(d, ws=w))
        stage_fns.append(lambda d=ds, w=w: _lib.hsa_layer_decode(d, ws=w))
        keep.append((g8, d, ds, w))
    torch.cuda.synchronize()
    us = rotating_us(fns, args.warmup, args.steps, stream)
    idx_ms = []
    for i in range(args.steps):
        stage_fns[i % len(stage_fns)]()
        stage[4].synchronize()
        idx_ms.append(stage[1].elapsed_time(stage[2]))
    for g8, d, ds, w in keep:
        assert _lib.hsa_workspace_status(w) == 0
    Di = runs[0].g.shape.Di
    nb = statistics.mean(layer_bytes(r.L, r.g.shape, 4, key_entry_bytes=Di + 4)["total"] for r in runs)
    ib = statistics.mean(layer_bytes(r.L, r.g.shape, 4, key_entry_bytes=Di + 4)["indexer"] for r in runs)
    it = statistics.mean(idx_ms)
    out["two_query_tokens"] = two_token_layer(args, peak)
    out["e4m3_keys"] = {
        "us": us, "algorithmic_bytes": nb, "achieved_gbs": nb / (us * 1e-6) / 1e9,
        "frac": nb / (us * 1e-6) / 1e9 / peak,
        "indexer_stage_us": it * 1000, "indexer_algorithmic_bytes": ib,
        "indexer_frac": ib / (it * 1e-3) / 1e9 / peak,
        "format": "E4M3 codes [rows, 128] + fp32 scale per row (amax / 448); queries "
                  "quantized per (sequence, head) in the kernel; tcgen05 kind::f8f6f4"}
    return out


def two_token_layer(args, peak, n=4):
    """The headline workload with two query tokens per sequence and step
    (speculative decoding with a one-layer MTP head: the current and a draft
    token verified together; the keys are streamed once for both), over n
    rotating layer states."""
    stream = torch.cuda.current_stream()
    fns, keep, nbytes = [], [], []
    for j in range(n):
        seed = synth.SEED["c4layer"] + 7919 * j
        L = synth.c4_lengths(seed, 64) + 1
        g = synth.filled_state(seed, 4, synth.FULL, L, device="cuda", name=f"mtp{j}", T=2)
        B, sh = L.numel(), g.shape
        out = torch.empty(B, 2, sh.Hq, sh.Dv, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, 2, sh.Hq, dtype=torch.float32, device="cuda")
        so = torch.empty_like(g.seq_len_in)
        d = _lib.layer_desc(g, out, lse, so)
        w = _lib.workspace(_lib.hsa_layer_decode_workspace_size(d))
        fns.append(lambda d=d, w=w: _lib.hsa_layer_decode(d, ws=w))
        keep.append((g, out, lse, so, d, w))
        nbytes.append(layer_bytes(L, sh, 4, T=2)["total"])
    us = rotating_us(fns, args.warmup, args.steps, stream)
    for *_, w in keep:
        assert _lib.hsa_workspace_status(w) == 0
    nb = statistics.mean(nbytes)
    return {"us_per_step": us, "us_per_token": us / 2, "tokens_per_step": 128,
            "algorithmic_bytes": nb, "achieved_gbs": nb / (us * 1e-6) / 1e9,
            "frac": nb / (us * 1e-6) / 1e9 / peak, "launches": _lib.hsa_layer_decode_launches(keep[0][4])}


def e2e_layer(runs, flush, warmup, steps):
    """The layer step through host buffers, over the given layer runs (step i
    on run i mod len(runs); with several runs, inputs larger than L2 and no
    flush, else the L2 flushed before each step): the step's inputs (q and the
    new token's rows) travel in one host-to-device copy (one pinned staging
    buffer, each input at a 256-byte-aligned offset) and its outputs in one
    device-to-host copy; the library reads and writes views of the device
    staging buffers.  (Uploading q on a second stream and making the attention
    wait for it with an event measured slower: the event wait ends the
    programmatic overlap of the attention with the indexer.)
    Returns (mean ms, h2d bytes, d2h bytes, host output of the last step of
    run 0, that run's device output)."""
    import copy as _copy

    def packed(tensors):
        offs, at = [], 0
        for t in tensors:
            offs.append(at)
            at += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, at

    stream = torch.cuda.current_stream()
    staged = []
    for r in runs:
        g = r.g
        names_in = ("q", "kv_new", "z_new") + (("ik_new", "iz_new", "iq", "w") if g.kind == 4 else ())
        t_in = [getattr(g, k) for k in names_in]
        offs_in, n_in = packed(t_in)
        dev_in = torch.empty(n_in, dtype=torch.uint8, device="cuda")
        host_in = torch.empty(n_in, dtype=torch.uint8).pin_memory()
        g2 = _copy.copy(g)
        for k, t, o in zip(names_in, t_in, offs_in):
            nb = t.numel() * t.element_size()
            host_in[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
            setattr(g2, k, dev_in[o:o + nb].view(t.dtype).view(t.shape))
        offs_out, n_out = packed([r.out, r.lse])
        dev_out = torch.empty(n_out, dtype=torch.uint8, device="cuda")
        out2 = dev_out[:r.out.numel() * 2].view(r.out.dtype).view(r.out.shape)
        lse2 = dev_out[offs_out[1]:offs_out[1] + r.lse.numel() * 4].view(r.lse.dtype).view(r.lse.shape)
        host_out = torch.empty(n_out, dtype=torch.uint8).pin_memory()
        desc = _lib.layer_desc(g2, out2, lse2, r.seq_out, None, r.scores)
        ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
        # bytes per step: the packed buffers as copied (inputs and alignment gaps)
        staged.append((dev_in, host_in, dev_out, host_out, desc, ws, n_in, n_out, out2))
    ts = []
    for i in range(warmup + steps):
        dev_in, host_in, dev_out, host_out, desc, ws, _, _, _ = staged[i % len(staged)]
        if len(staged) == 1:
            flush(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_in.copy_(host_in, non_blocking=True)
        _lib.hsa_layer_decode(desc, ws=ws)
        host_out.copy_(dev_out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= warmup:
            ts.append(a.elapsed_time(b))
    for st in staged:
        assert _lib.hsa_workspace_status(st[5]) == 0
    h2d, d2h = staged[0][6], staged[0][7]
    host_o = staged[0][3][:runs[0].out.numel() * 2].view(runs[0].out.dtype).view(runs[0].out.shape)
    return statistics.mean(ts), h2d, d2h, host_o, staged[0][8]


NSTATES = 4


class LayerRun:
    """One layer state of the bench workload with its outputs, descriptors
    (plain and with stage events) and workspace."""

    def __init__(self, L, g, stage_events=None):
        self.L, self.g = L, g
        self.out, self.lse, self.seq_out, _, self.scores = layer_outputs(g)
        # a decode loop needs the attention output, not the index list
        self.desc = _lib.layer_desc(g, self.out, self.lse, self.seq_out, None, self.scores)
        self.desc_stages = None
        if stage_events is not None:
            self.desc_stages = _lib.layer_desc(g, self.out, self.lse, self.seq_out, None,
                                               self.scores, stage_events=stage_events)
        self.ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(self.desc))
        self.nbytes = layer_bytes(L, g.shape, g.kind)

    def step(self, stages=False):
        _lib.hsa_layer_decode(self.desc_stages if stages else self.desc, ws=self.ws)


def layer_runs(rank, n=NSTATES, stage_events=None):
    """n layer states of the bench workload (the rank's own first), each ~1.7
    GB of pools and rings: together far larger than L2."""
    runs = []
    for j in range(n):
        if j == 0:
            L, g = build_workload(rank)
        else:
            seed = synth.SEED["c4layer"] + 1000 * rank + 7919 * j
            L = synth.c4_lengths(seed, 64)
            g = synth.filled_state(seed, 4, synth.FULL, L, device="cuda", name=f"layer{j}")
        runs.append(LayerRun(L, g, stage_events))
    return runs


def measure_c4layer(args, rank, local, dist):
    """The headline: one C4 layer step of the bench workload (see the module
    docstring), device-timed and end to end.  Step i works on layer state i
    mod 4 (each larger than L2, 368 MB of algorithmic traffic per step), with
    no L2 flush: like consecutive layers of a decode step, each step's data is
    cold while the kernels' code and small state stay in L2.  The same step
    with the L2 flushed before it (state 0 every time) is reported beside it.
    On rank 0 also the other configurations, the 60-layer CUDA graph and the
    oracle baseline."""
    _lib.load(build_if_missing=True)
    stream = torch.cuda.current_stream()
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in stage:
        e.record(stream)          # the events exist from here on
    # the timed steps run without stage events: an event recorded between two
    # kernels stops the next one from being scheduled while the previous runs
    runs = layer_runs(rank, stage_events=[e.cuda_event for e in stage])
    launches = _lib.hsa_layer_decode_launches(runs[0].desc)
    flush = L2Flush()
    total_bytes = statistics.mean(r.nbytes["total"] for r in runs)
    nbytes = {k: statistics.mean(r.nbytes[k] for r in runs) for k in runs[0].nbytes}

    for i in range(max(args.warmup, NSTATES)):
        runs[i % NSTATES].step()
    torch.cuda.synchronize()
    for r in runs:
        assert _lib.hsa_workspace_status(r.ws) == 0

    # ------------------------------------------------ device-timed region
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            ev0[i].record(stream)
            runs[i % NSTATES].step()
            ev1[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(dist)
    ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ev0, ev1))
    # the same step with the L2 flushed before it (state 0)
    ms_flushed = statistics.mean(timed(lambda: runs[0].step(), flush, 2, args.steps, stream))
    # per-kernel durations: the same rotation with an event between kernels
    stage_ms = []
    for i in range(args.steps):
        runs[i % NSTATES].step(stages=True)
        stage[4].synchronize()                  # stage events are reused: read them now
        stage_ms.append([stage[j].elapsed_time(stage[j + 1]) for j in range(4)])
    stage_mean = np.array(stage_ms).mean(axis=0)  # append, indexer, top-k, attention (ms)
    for r in runs:
        assert _lib.hsa_workspace_status(r.ws) == 0

    e2e_ms, h2d, d2h, host_o, dev_o = e2e_layer(runs, flush, args.warmup, args.steps)
    torch.cuda.synchronize()
    runs[0].step()
    torch.cuda.synchronize()
    assert torch.equal(host_o, runs[0].out.cpu())

    extra = {}
    peak, peak_kind = measured_peaks()
    if rank == 0 and not args.no_extra:
        extra["layer_variants"] = layer_variants(args, runs, peak)
        if args.layers > 0:
            extra["multi_layer_graph"] = multi_layer_graph(args, flush, runs)
        extra["topk_rows_per_s"] = bench_topk(flush, args)
        extra["compress"] = bench_compress(flush, args)
        extra["longctx"] = bench_longctx(flush, args)
    cpu = None
    if rank == 0 and args.cpu_budget > 0:
        run, threads, busy = oracle_layer_runner(runs[0].g)
        sec, calls = time_oracle(run, args.cpu_budget)
        cpu = {"value": sec * 1e6, "unit": "us", "cores": threads, "kind": "oracle",
               "sample": f"the whole 64-sequence layer step (state 0), {calls} calls "
                         f"(~{args.cpu_budget:.0f} s budget), mean",
               "threads_busy_by_stage": busy}

    idx_ms = float(stage_mean[1])
    achieved = nbytes["indexer"] / (idx_ms * 1e-3) / 1e9
    layer_gbs = total_bytes / (ms * 1e-3) / 1e9
    line = base_line(args, 1, METRIC, "us", False, WORKLOAD, ms * 1000)
    line["config"].update({
        "l2": f"inputs larger than L2: step i on layer state i mod {NSTATES} (each ~1.7 GB, "
              f"{total_bytes / 1e6:.0f} MB of algorithmic traffic per step), no flush; "
              f"l2_flushed_us: the same step on state 0 after {L2_NOTE}",
        "sum_c4_entries": int((runs[0].L // 4).sum()), "seed": synth.SEED["c4layer"],
        "states": NSTATES,
        "outputs": "attention output and log-sum-exp (the top-k index list is not requested)"})
    line.update({
        "l2_flushed_us": ms_flushed * 1000,
        "roofline": {"bound": "hbm", "kernel": "indexer_kernel (tcgen05 scores)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)",
                     "traffic": indexer_traffic(), "algorithmic_bytes": nbytes["indexer"],
                     "launch_us": idx_ms * 1000},
        "layer_roofline": {"algorithmic_bytes": total_bytes, "achieved_gbs": layer_gbs,
                           "frac": layer_gbs / peak},
        "stage_rooflines": {
            name: {"algorithmic_bytes": nbytes[key], "stage_us": stage_mean[j] * 1000,
                   "achieved_gbs": nbytes[key] / (stage_mean[j] * 1e-3) / 1e9,
                   "frac": nbytes[key] / (stage_mean[j] * 1e-3) / 1e9 / peak}
            for name, key, j in (("indexer", "indexer", 1),
                                 ("selection + attention (+ split merge)", "attention", 3))},
        "stage_us": {"append_compress": stage_mean[0] * 1000, "indexer": stage_mean[1] * 1000,
                     "topk (own kernels only; fused into the attention otherwise)":
                         stage_mean[2] * 1000,
                     "attention": stage_mean[3] * 1000},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_ms * 1000, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": wall,
    })
    line.update(extra)
    B = runs[0].L.numel()
    return {"ms": ms, "e2e_ms": e2e_ms, "line": line, "units_per_step": 1,
            "tokens_per_step": B, "throughput_unit": "decode tokens/s through one layer"}


def run_profile(ctx=None):
    """Two layer steps of the bench workload (the first warms up), for ncu."""
    _lib.load(build_if_missing=True)
    L, g = build_workload(0, ctx)
    out, lse, seq_out, _, scores = layer_outputs(g)
    # as the bench's step: the attention output and log-sum-exp, no index list
    desc = _lib.layer_desc(g, out, lse, seq_out, None, scores)
    ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
    for _ in range(2):
        _lib.hsa_layer_decode(desc, ws=ws)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    print(json.dumps({"profile": "ok", "sum_c4_entries": int((L // 4).sum())}))


def run_profile_topk():
    """Two top-k calls on the standalone workload (the first warms up), for ncu."""
    _lib.load(build_if_missing=True)
    x, offs = topk_inputs()
    idx = torch.empty(64, 512, dtype=torch.int32, device="cuda")
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(64, x.numel(), 512))
    for _ in range(2):
        _lib.hsa_topk(x, offs, 512, idx=idx, ws=ws, with_vals=False)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    print(json.dumps({"profile": "ok", "scores": int(x.numel())}))


def run_profile_compress(S=4):
    """Two compressor calls at each ratio (r = 4, then r = 128; the first of
    each warms up) on S sequences of the standalone shape (65,536 x 512: 537 MB
    of kv and z at S = 4, larger than L2), for ncu."""
    _lib.load(build_if_missing=True)
    seed = synth.SEED["compress"]
    kv = synth.normal_bf16(seed, "compress.kv", (S, 65536, 512), device="cuda")
    z = synth.normal_bf16(seed, "compress.z", (S, 65536, 512), device="cuda")
    for r in (4, 128):
        b = synth.normal(seed, f"compress.b{r}", (r, 512), std=0.5, device="cuda")
        out = torch.empty(S, 65536 // r, 512, dtype=torch.bfloat16, device="cuda")
        for _ in range(2):
            _lib.hsa_compress(kv, z, b, r, out=out)
    torch.cuda.synchronize()
    print(json.dumps({"profile": "ok", "sequences": S}))


def multi_layer_graph(args, flush, runs, iters=10):
    """A decode step over `args.layers` C4 layers (the bench's shapes; layer i
    works on state i mod len(runs), each larger than L2) captured once in a
    CUDA graph: us per layer of the replayed step, next to the same layers
    launched one call at a time; the L2 is flushed before each step."""
    descs = [runs[i % len(runs)] for i in range(args.layers)]

    def eager():
        for r in descs:
            r.step()

    for _ in range(3):
        eager()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        eager()
    times = {"graph": [], "eager": []}
    for i in range(3 + iters):
        for mode in ("graph", "eager"):
            flush(i)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            if mode == "graph":
                graph.replay()
            else:
                eager()
            b.record()
            b.synchronize()
            if i >= 3:
                times[mode].append(a.elapsed_time(b))
    for r in runs:
        assert _lib.hsa_workspace_status(r.ws) == 0
    per = {m: statistics.mean(v) * 1000 / args.layers for m, v in times.items()}
    del graph
    torch.cuda.empty_cache()
    return {"layers": args.layers, "states": len(runs), "us_per_layer_graph": per["graph"],
            "us_per_layer_eager": per["eager"],
            "note": f"C4 layers of the bench workload, layer i on state i mod {len(runs)}; L2 "
                    "flushed before each step, not between layers"}


# ----------------------------------------------------------------------------- other configurations

TOPK_METRIC = "top-512 rows/s (Lightning TopK, 64 rows x 262,144 fp32)"
TOPK_WORKLOAD = "64 x 262,144 fp32 N(0,1), 5% of entries copies of others (ties), k=512"
COMPRESS_METRIC = "us per Flash Compressor call (32 x 65,536 tokens x 512 channels, r=4)"
COMPRESS_WORKLOAD = ("Flash Compressor: 32 sequences x 65,536 tokens x 512 channels, kv and z bf16 "
                     "N(0,1), b fp32 N(0,0.5^2), bf16 output; r=4 (headline) and r=128")
LONG_METRIC = "us per decode layer (C4+SWA, 1M ctx, batch 4)"
LONG_WORKLOAD = ("1M-token pair: B=4, L=1,048,576 (the step completes a 4- and a 128-token "
                 "block), Hq=64, Dqk=576, Dv=512, window 128; (a) C4: indexer 8x128, top-512 "
                 "over 262,144 entries; (b) C128: dense over 8,192 entries")


def topk_inputs(device="cuda"):
    x = synth.topk_scores(synth.SEED["topk"], 64, 262144, 0.05, device=device).reshape(-1)
    offs = torch.arange(65, dtype=torch.int64, device=device) * 262144
    return x, offs


def oracle_topk_runner():
    import oracle
    threads = oracle_threads()
    x, offs = topk_inputs("cuda" if torch.cuda.is_available() else "cpu")
    xs, os_ = x.cpu().numpy(), offs.cpu().numpy()

    def run():
        oracle.topk(xs, os_, 512, threads=threads)

    return run, threads, {"topk": min(threads, 64)}, "all 64 rows per timed step"


def bench_topk(flush, args, iters=20):
    """Standalone Lightning TopK on 64 rows x 262,144 fp32 (5% copied entries),
    k=512: rows per second, L2 flushed before each launch."""
    x, offs = topk_inputs()
    idx = torch.empty(64, 512, dtype=torch.int32, device="cuda")
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(64, x.numel(), 512))
    ts = timed(lambda: _lib.hsa_topk(x, offs, 512, idx=idx, ws=ws, with_vals=False), flush, 3, iters)
    assert _lib.hsa_workspace_status(ws) == 0
    ms = statistics.mean(ts)
    peak, _ = measured_peaks()
    gbs = x.numel() * 4 / (ms * 1e-3) / 1e9
    res = {"value": 64 / (ms * 1e-3), "unit": "rows/s", "us_per_call": ms * 1000,
           "config": "64 x 262,144 fp32, 5% copied entries, k=512",
           "algorithmic_bytes": x.numel() * 4 + 64 * 512 * 4,
           "achieved_gbs": gbs, "frac_of_hbm": gbs / peak}
    if args.cpu_budget > 0:
        run, threads, busy, sample = oracle_topk_runner()
        sec, calls = time_oracle(run, 0.0)
        res["cpu_baseline"] = {"value": 64 / sec, "unit": "rows/s", "cores": threads,
                               "kind": "oracle", "sample": sample, "threads_busy_by_stage": busy}
    return res


def measure_topk_line(args, rank, local, dist):
    _lib.load(build_if_missing=True)
    flush = L2Flush()
    x, offs = topk_inputs()
    idx = torch.empty(64, 512, dtype=torch.int32, device="cuda")
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(64, x.numel(), 512))
    fn = lambda: _lib.hsa_topk(x, offs, 512, idx=idx, ws=ws, with_vals=False)
    barrier(dist)
    with ClockSampler(local) as clocks:
        ts = timed(fn, flush, args.warmup, args.steps)
    barrier(dist)
    ms = statistics.mean(ts)
    # end to end: scores from pinned host memory, indices back
    xh = x.cpu().pin_memory()
    ih = torch.empty(64, 512, dtype=torch.int32).pin_memory()
    xd = torch.empty_like(x)

    def e2e():
        xd.copy_(xh, non_blocking=True)
        _lib.hsa_topk(xd, offs, 512, idx=idx, ws=ws, with_vals=False)
        ih.copy_(idx, non_blocking=True)

    e2e_ms = statistics.mean(timed(e2e, flush, args.warmup, args.steps))
    assert torch.equal(ih, idx.cpu())
    peak, peak_kind = measured_peaks()
    nb = x.numel() * 4 + 64 * 512 * 4
    gbs = nb / (ms * 1e-3) / 1e9
    line = base_line(args, 1, TOPK_METRIC, "rows/s", True, TOPK_WORKLOAD, 64 / (ms * 1e-3))
    line["dtype"] = "u32"
    line["config"]["l2"] = L2_NOTE
    cpu = None
    if rank == 0 and args.cpu_budget > 0:
        run, threads, busy, sample = oracle_topk_runner()
        sec, calls = time_oracle(run, min(args.cpu_budget, 5.0))
        cpu = {"value": 64 / sec, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": sample, "threads_busy_by_stage": busy}
    launches = 1  # one launch per call (clustered rows or chunked rows)
    line.update({"roofline": {"bound": "hbm", "kernel": "topk_chunk_kernel",
                              "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                              "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)",
                              "traffic": profile_traffic("topk_chunk_64x262144_traffic.json", TOPK_SOURCES),
                              "algorithmic_bytes": nb, "launch_us": ms * 1000},
                 "cpu_baseline": cpu,
                 "e2e": {"value": None, "unit": "rows/s", "h2d_bytes_per_step": x.numel() * 4,
                         "d2h_bytes_per_step": 64 * 512 * 4},
                 "gpu_launches": launches * args.steps, "clocks": clocks.summary()})
    return {"ms": ms, "e2e_ms": e2e_ms, "line": line, "units_per_step": 64,
            "throughput_unit": "rows/s"}


def compress_inputs(r, device="cuda"):
    seed = synth.SEED["compress"]
    S, T, C = 32, 65536, 512
    kv = synth.normal_bf16(seed, "compress.kv", (S, T, C), device=device)
    z = synth.normal_bf16(seed, "compress.z", (S, T, C), device=device)
    b = synth.normal(seed, f"compress.b{r}", (r, C), std=0.5, device=device)
    return kv, z, b


def compress_bytes(S, T, C, r):
    return 2 * S * T * C * 2 + S * (T // r) * C * 2 + r * C * 4


def oracle_compress_runner(r, kv=None, z=None, b=None, seqs=2):
    """The oracle compressor on `seqs` of the 32 sequences; returns (run,
    threads, busy, sample, scale to the full 32)."""
    import oracle
    threads = oracle_threads()
    if kv is None:
        kv, z, b = compress_inputs(r, "cuda" if torch.cuda.is_available() else "cpu")
    kvs, zs, bs = _bits(kv[:seqs]), _bits(z[:seqs]), b.cpu().numpy()

    def run():
        oracle.compress(kvs, zs, bs, r, threads=threads)

    nblk = seqs * (kv.shape[1] // r)
    return (run, threads, {"compress": min(threads, nblk)},
            f"{seqs} of the 32 sequences per timed step, scaled x{32 // seqs}", 32 / seqs)


def bench_compress(flush, args, iters=5):
    """Flash Compressor standalone, 32 x 65,536 x 512, r = 4 and r = 128, bf16 output."""
    peak, _ = measured_peaks()
    res = {}
    kv = z = None
    for r in (4, 128):
        if kv is None:
            kv, z, b = compress_inputs(r)
        else:
            b = synth.normal(synth.SEED["compress"], f"compress.b{r}", (r, 512), std=0.5,
                             device="cuda")
        out = torch.empty(32, 65536 // r, 512, dtype=torch.bfloat16, device="cuda")
        ms = statistics.mean(timed(lambda: _lib.hsa_compress(kv, z, b, r, out=out), flush, 2, iters))
        nb = compress_bytes(32, 65536, 512, r)
        gbs = nb / (ms * 1e-3) / 1e9
        ent = {"us": ms * 1000, "algorithmic_bytes": nb, "achieved_gbs": gbs, "frac": gbs / peak,
               "roofline_us_at_peak": nb / (peak * 1e9) * 1e6}
        if args.cpu_budget > 0:
            run, threads, busy, sample, scale = oracle_compress_runner(r, kv, z, b)
            sec, calls = time_oracle(run, 0.0)
            ent["cpu_baseline"] = {"value": sec * scale * 1e6, "unit": "us", "cores": threads,
                                   "kind": "oracle", "sample": sample,
                                   "threads_busy_by_stage": busy}
        res[f"r{r}"] = ent
        del out
    del kv, z
    torch.cuda.empty_cache()
    res["config"] = COMPRESS_WORKLOAD
    return res


def measure_compress_line(args, rank, local, dist):
    _lib.load(build_if_missing=True)
    flush = L2Flush()
    kv, z, b = compress_inputs(4)
    out = torch.empty(32, 16384, 512, dtype=torch.bfloat16, device="cuda")
    fn = lambda: _lib.hsa_compress(kv, z, b, 4, out=out)
    barrier(dist)
    with ClockSampler(local) as clocks:
        ts = timed(fn, flush, args.warmup, args.steps)
    barrier(dist)
    ms = statistics.mean(ts)
    # end to end: kv and z from pinned host memory, the compressed rows back
    kvh, zh = kv.cpu().pin_memory(), z.cpu().pin_memory()
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e():
        kv.copy_(kvh, non_blocking=True)
        z.copy_(zh, non_blocking=True)
        _lib.hsa_compress(kv, z, b, 4, out=out)
        oh.copy_(out, non_blocking=True)

    e2e_ms = statistics.mean(timed(e2e, flush, 1, max(2, args.steps // 5)))
    peak, peak_kind = measured_peaks()
    nb = compress_bytes(32, 65536, 512, 4)
    gbs = nb / (ms * 1e-3) / 1e9
    line = base_line(args, 1, COMPRESS_METRIC, "us", False, COMPRESS_WORKLOAD, ms * 1000)
    line["config"]["l2"] = L2_NOTE
    cpu = None
    if rank == 0 and args.cpu_budget > 0:
        run, threads, busy, sample, scale = oracle_compress_runner(4, kv, z, b)
        sec, calls = time_oracle(run, min(args.cpu_budget, 5.0))
        cpu = {"value": sec * scale * 1e6, "unit": "us", "cores": threads, "kind": "oracle",
               "sample": sample, "threads_busy_by_stage": busy}
    line.update({"roofline": {"bound": "hbm", "kernel": "compress_kernel", "achieved": gbs,
                              "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                              "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)", "traffic": None,
                              "algorithmic_bytes": nb, "launch_us": ms * 1000},
                 "cpu_baseline": cpu,
                 "e2e": {"value": None, "unit": "us", "h2d_bytes_per_step": 2 * kv.numel() * 2,
                         "d2h_bytes_per_step": out.numel() * 2},
                 "gpu_launches": args.steps, "clocks": clocks.summary()})
    if rank == 0:
        line["r128"] = bench_compress(flush, args)["r128"]
    return {"ms": ms, "e2e_ms": e2e_ms, "line": line, "units_per_step": 1,
            "tokens_per_step": 32 * 65536, "throughput_unit": "tokens compressed/s"}


def bench_layer_state(L, g, flush, warmup, steps, cpu_budget, clocks=None, dist=None):
    """Device time, algorithmic bytes, end-to-end time and oracle baseline of
    one layer step of state g (clocks, if given, is sampled around the
    device-timed steps only, which barriers bracket)."""
    out, lse, seq_out, idx, scores = layer_outputs(g)
    desc = _lib.layer_desc(g, out, lse, seq_out, idx, scores)
    ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
    fn = lambda: _lib.hsa_layer_decode(desc, ws=ws)
    for i in range(warmup):
        flush(i)
        fn()
    torch.cuda.synchronize()
    barrier(dist)
    if clocks is not None:
        with clocks:
            ts = timed(fn, flush, 0, steps)
    else:
        ts = timed(fn, flush, 0, steps)
    barrier(dist)
    ms = statistics.mean(ts)
    assert _lib.hsa_workspace_status(ws) == 0
    peak, _ = measured_peaks()
    nb = layer_bytes(L, g.shape, g.kind)
    gbs = nb["total"] / (ms * 1e-3) / 1e9
    ent = {"us": ms * 1000, "algorithmic_bytes": nb["total"], "achieved_gbs": gbs,
           "frac": gbs / peak, "launches": _lib.hsa_layer_decode_launches(desc),
           "e2e": None}
    run = LayerRun(L, g)
    e2e_ms, h2d, d2h, _, _ = e2e_layer([run], flush, warmup, steps)
    ent["e2e"] = {"value": e2e_ms * 1000, "unit": "us", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h}
    if cpu_budget > 0:
        run, threads, busy = oracle_layer_runner(g)
        sec, calls = time_oracle(run, 0.0)
        ent["cpu_baseline"] = {"value": sec * 1e6, "unit": "us", "cores": threads,
                               "kind": "oracle", "sample": "the whole batch-4 layer step",
                               "threads_busy_by_stage": busy}
    return ent, ms, e2e_ms


def bench_longctx(flush, args, steps=10):
    res = {"config": LONG_WORKLOAD}
    for kind in (4, 128):
        L, g = longctx_workload(kind)
        ent, _, _ = bench_layer_state(L, g, flush, 3, steps, args.cpu_budget)
        res["c4" if kind == 4 else "c128"] = ent
        del g
        torch.cuda.empty_cache()
    return res


def measure_longctx_line(args, rank, local, dist):
    _lib.load(build_if_missing=True)
    flush = L2Flush()
    L, g = longctx_workload(4, rank)
    clocks = ClockSampler(local)
    ent, ms, e2e_ms = bench_layer_state(L, g, flush, args.warmup, args.steps,
                                        args.cpu_budget if rank == 0 else 0, clocks, dist)
    del g
    torch.cuda.empty_cache()
    peak, peak_kind = measured_peaks()
    line = base_line(args, 1, LONG_METRIC, "us", False, LONG_WORKLOAD, ms * 1000)
    line["config"]["l2"] = L2_NOTE
    line.update({"layer_roofline": {"algorithmic_bytes": ent["algorithmic_bytes"],
                                    "achieved_gbs": ent["achieved_gbs"], "frac": ent["frac"]},
                 "roofline": {"bound": "hbm", "kernel": "whole C4 layer step", "achieved":
                              ent["achieved_gbs"], "peak": peak, "unit": "GB/s",
                              "frac": ent["frac"], "peak_kind": f"{peak_kind} hbm_gbs",
                              "traffic": None, "algorithmic_bytes": ent["algorithmic_bytes"]},
                 "cpu_baseline": ent.get("cpu_baseline"), "e2e": ent["e2e"],
                 "gpu_launches": ent["launches"] * args.steps, "clocks": clocks.summary()})
    if rank == 0:
        L2_, g2 = longctx_workload(128)
        line["c128"], _, _ = bench_layer_state(L2_, g2, flush, 3, args.steps, args.cpu_budget)
    return {"ms": ms, "e2e_ms": e2e_ms, "line": line, "units_per_step": 1,
            "tokens_per_step": 4, "throughput_unit": "decode tokens/s through one layer"}


INDEXER_SOURCES = ("indexer.cu", "tc.cuh", "common.cuh")
TOPK_SOURCES = ("topk.cu", "select_core.cuh", "tc.cuh", "common.cuh")


def profile_traffic(name, sources):
    """DRAM bytes per launch from a committed ncu summary under profiles/, if it
    was taken on the current source of the kernel (else null)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, "hybrid_sparse_attention_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


def indexer_traffic():
    return profile_traffic("indexer_c4layer_traffic.json", INDEXER_SOURCES)


if __name__ == "__main__":
    main()
