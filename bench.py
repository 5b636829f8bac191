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

Prints one JSON line (rank 0).  Under torchrun with N > 1 every rank runs an
independent replica of the workload (its own seed): weak scaling, no data-path
collective; the time is the maximum over ranks.
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


def layer_bytes(L, shape):
    """Algorithmic HBM bytes of one C4 layer step (each byte the method must
    move, counted once): indexer keys, score write + read, the gathered window
    and top-k rows, q, o, the index list, plus the new-token append and the
    4-row block reads/writes of the sequences whose block completes."""
    L = L.to(torch.int64)
    n4 = L // 4
    B = L.numel()
    D, Di = shape.Dqk, shape.Di
    keys = int(n4.sum()) * Di * 2
    iq_w = B * shape.Hi * (Di * 2 + 4)
    scores = 2 * int(n4.sum()) * 4
    rows = int((torch.clamp(L, max=shape.W) + torch.clamp(n4, max=shape.k)).sum())
    gather = rows * D * 2
    q = B * shape.Hq * D * 2
    o = B * shape.Hq * shape.Dv * 2 + B * shape.Hq * 4
    idx = 2 * B * shape.k * 4
    append = B * (D * 2 * 2 + D * 2 * 3 + Di * 2 * 2 + Di * 2 * 2)   # read new rows, write rings
    ncomp = int((L % 4 == 0).sum())
    compress = ncomp * (4 * 2 * (D + Di) * 2 + (D + Di) * 2)
    indexer = keys + iq_w + int(n4.sum()) * 4
    total = keys + iq_w + scores + gather + q + o + idx + append + compress
    attention = gather + q + o + idx // 2
    topk = int(n4.sum()) * 4 + idx // 2
    return {"total": total, "indexer": indexer, "keys": keys, "gather": gather,
            "attention": attention, "topk": topk}


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


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
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

def sample_state(g, seqs):
    """numpy copy (oracle input) of sequences `seqs` of a GPU layer state."""
    offs = g.pool_offsets.cpu()
    bits = lambda t: t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()
    kv = torch.cat([g.kv_pool[int(offs[b]):int(offs[b + 1])] for b in seqs])
    key = torch.cat([g.key_pool[int(offs[b]):int(offs[b + 1])] for b in seqs])
    caps = torch.tensor([int(offs[b + 1] - offs[b]) for b in seqs], dtype=torch.int64)
    new_offs = torch.zeros(len(seqs) + 1, dtype=torch.int64)
    new_offs[1:] = torch.cumsum(caps, 0)
    sel = torch.tensor(seqs, device=g.q.device)
    s = {"kind": g.kind, "ratio": g.ratio, "Dv": g.shape.Dv, "k": g.shape.k,
         "scale": g.shape.scale, "pool_offsets": new_offs.numpy(),
         "seq_len_in": g.seq_len_in[sel].cpu().numpy(), "kv_pool": bits(kv), "key_pool": bits(key),
         "b_kv": g.b_kv.cpu().numpy(), "b_ik": g.b_ik.cpu().numpy(),
         "w": g.w[sel].cpu().numpy()}
    for name in ("swa", "kv_ring", "z_ring", "ik_ring", "iz_ring", "kv_new", "z_new", "ik_new",
                 "iz_new", "q", "iq"):
        s[name] = bits(getattr(g, name)[sel])
    return s


def oracle_layer_time(g, budget_s, per_call=4):
    """Times the oracle layer step over successive sequence groups until the
    budget is spent; returns (us per full 64-sequence layer, sequences, threads)."""
    import oracle
    oracle.build()
    threads = oracle.hardware_threads()
    B = g.seq_len_in.numel()
    done, spent = 0, 0.0
    while done < B and (spent < budget_s or done == 0):
        seqs = list(range(done, min(B, done + per_call)))
        s = sample_state(g, seqs)
        t0 = time.perf_counter()
        oracle.layer_decode(s, threads=threads)
        spent += time.perf_counter() - t0
        done += len(seqs)
    return spent / done * B * 1e6, done, threads


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="hsa", choices=["hsa", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline (0: skip)")
    ap.add_argument("--layers", type=int, default=60,
                    help="layers in the CUDA-graph multi-layer step measurement (0: skip)")
    ap.add_argument("--no-topk", action="store_true",
                    help="skip the standalone top-k rows/s measurement")
    ap.add_argument("--profile", action="store_true",
                    help="profiling run: build the workload, run two layer steps, exit")
    ap.add_argument("--profile-ctx", type=int, nargs=2, default=None, metavar=("LO", "HI"),
                    help="with --profile: context lengths ~ U[LO, HI] instead of the bench's "
                         "(a smaller case of the same layer for multi-pass ncu captures)")
    args = ap.parse_args()
    world, rank, local, dist = dist_setup()
    torch.cuda.set_device(local)
    if args.impl == "reference":
        run_reference(args, world, rank, dist)
    elif args.profile:
        run_profile(args.profile_ctx)
    else:
        run_hsa(args, world, rank, local, dist)
    if dist is not None:
        dist.destroy_process_group()


def build_workload(rank, ctx=None):
    seed = synth.SEED["c4layer"] + 1000 * rank
    L = synth.c4_lengths(seed, 64) if ctx is None else synth.c4_lengths(seed, 64, ctx[0], ctx[1])
    g = synth.filled_state(seed, 4, synth.FULL, L, device="cuda")
    return L, g


def run_reference(args, world, rank, dist):
    """The oracle (plain CPU C++), as it stands, on the host cores: each step is
    one bounded sample of the same workload scaled to a full layer."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    L, g = build_workload(0)
    threads = oracle.hardware_threads()
    per_step = 2
    for i in range(args.warmup):
        oracle.layer_decode(sample_state(g, [i % 64]), threads=threads)
    times = []
    for i in range(args.steps):
        seqs = [(per_step * i + j) % 64 for j in range(per_step)]
        s = sample_state(g, seqs)
        t0 = time.perf_counter()
        oracle.layer_decode(s, threads=threads)
        times.append((time.perf_counter() - t0) / per_step * 64 * 1e6)
    us = statistics.mean(times)
    sample = f"{per_step} of the 64 sequences per step (rotating), scaled x{64 // per_step}"
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1000,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": us, "unit": "us", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_hsa(args, world, rank, local, dist):
    _lib.load(build_if_missing=True)
    shape = synth.FULL
    L, g = build_workload(rank)
    B = L.numel()
    stream = torch.cuda.current_stream()
    out = torch.empty(B, shape.Hq, shape.Dv, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, shape.Hq, dtype=torch.float32, device="cuda")
    seq_out = torch.empty_like(g.seq_len_in)
    idx = torch.empty(B, shape.k, dtype=torch.int32, device="cuda")
    scores = torch.empty(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in stage:
        e.record(stream)          # the events exist from here on
    # the timed steps run without stage events: an event recorded between two
    # kernels stops the next one from being scheduled while the previous runs
    desc = _lib.layer_desc(g, out, lse, seq_out, idx, scores)
    desc_stages = _lib.layer_desc(g, out, lse, seq_out, idx, scores,
                                  stage_events=[e.cuda_event for e in stage])
    ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
    launches = _lib.hsa_layer_decode_launches(desc)
    flush = L2Flush()
    nbytes = layer_bytes(L, shape)

    def step(d=desc):
        _lib.hsa_layer_decode(d, ws=ws)

    for _ in range(args.warmup):
        flush(0)
        step()
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0

    # ------------------------------------------------ device-timed region
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush(i)                            # evict the previous step's data from L2
            ev0[i].record(stream)
            step()
            ev1[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(dist)
    t_layer = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    # per-kernel durations: the same steps again with an event between kernels
    stage_ms = []
    for i in range(args.steps):
        flush(i)
        step(desc_stages)
        stage[4].synchronize()                  # stage events are reused: read them now
        stage_ms.append([stage[j].elapsed_time(stage[j + 1]) for j in range(4)])
    ms = statistics.mean(t_layer)
    ms_max = max_over_ranks(ms, dist)
    st = np.array(stage_ms)
    stage_mean = st.mean(axis=0)                # append, indexer, top-k, attention (ms)
    assert _lib.hsa_workspace_status(ws) == 0

    # ------------------------------------------------ end to end: host buffers
    # The step's small inputs travel in one host-to-device copy (one pinned
    # staging buffer, each input at a 256-byte-aligned offset) and its outputs
    # in one device-to-host copy; the library reads and writes views of the
    # device staging buffers.  q (4.7 MB, read only by the attention) is copied
    # on a second stream inside the timed region and the layer waits for it
    # right before the attention (the descriptor's q-ready event), so its
    # upload overlaps the append, indexer and top-k.
    import copy as _copy

    def packed(tensors):
        offs, at = [], 0
        for t in tensors:
            offs.append(at)
            at += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, at

    names_in = ("kv_new", "z_new", "ik_new", "iz_new", "iq", "w")
    t_in = [getattr(g, k) for k in names_in]
    offs_in, n_in = packed(t_in)
    dev_in = torch.empty(n_in, dtype=torch.uint8, device="cuda")
    host_in = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    g2 = _copy.copy(g)
    for k, t, o in zip(names_in, t_in, offs_in):
        nb = t.numel() * t.element_size()
        host_in[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
        setattr(g2, k, dev_in[o:o + nb].view(t.dtype).view(t.shape))
    offs_out, n_out = packed([out, lse])
    dev_out = torch.empty(n_out, dtype=torch.uint8, device="cuda")
    out2 = dev_out[:out.numel() * 2].view(out.dtype).view(out.shape)
    lse2 = dev_out[offs_out[1]:offs_out[1] + lse.numel() * 4].view(lse.dtype).view(lse.shape)
    host_out = torch.empty(n_out, dtype=torch.uint8).pin_memory()
    q_host = g.q.cpu().pin_memory()
    g2.q = torch.empty_like(g.q)
    side = torch.cuda.Stream()
    q_ready = torch.cuda.Event()
    q_ready.record(side)                        # the event exists before its handle is taken
    desc_e2e = _lib.layer_desc(g2, out2, lse2, seq_out, idx, scores,
                               q_ready_event=q_ready.cuda_event)
    h2d, d2h = n_in + q_host.numel() * q_host.element_size(), n_out
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        side.wait_event(a)
        with torch.cuda.stream(side):
            g2.q.copy_(q_host, non_blocking=True)
            q_ready.record(side)
        dev_in.copy_(host_in, non_blocking=True)
        step(desc_e2e)
        host_out.copy_(dev_out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e = max_over_ranks(statistics.mean(e2e_ms), dist)
    assert torch.equal(host_out[:out.numel() * 2].view(out.dtype).view(out.shape), out.cpu())

    # ------------------------------------------------ a 60-layer step in one CUDA graph
    multi = multi_layer_graph(args, flush) if rank == 0 and args.layers > 0 else None

    # ------------------------------------------------ standalone top-k (rows / s)
    topk = topk_rows_per_s(flush) if rank == 0 and not args.no_topk else None

    # ------------------------------------------------ CPU baseline: the oracle
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        us_cpu, nseq, threads = oracle_layer_time(g, args.cpu_budget)
        cpu = {"value": us_cpu, "unit": "us", "cores": threads, "kind": "oracle",
               "sample": f"oracle layer step on {nseq} of the 64 sequences "
                         f"(groups of 4, ~{args.cpu_budget:.0f} s budget), scaled to 64"}

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    idx_ms = float(stage_mean[1])
    achieved = nbytes["indexer"] / (idx_ms * 1e-3) / 1e9
    layer_gbs = nbytes["total"] / (ms * 1e-3) / 1e9
    traffic = indexer_traffic()
    line = {
        "metric": METRIC,
        "value": ms_max * 1000 / world,
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                   "l2": f"{L2_FLUSH_BYTES >> 20} MiB written, then {L2_FLUSH_BYTES >> 21} MiB read, "
                         "before every step, outside the timed events (L2 cold and clean)",
                   "sum_c4_entries": int((L // 4).sum()), "seed": synth.SEED["c4layer"]},
        "roofline": {"bound": "hbm", "kernel": "indexer_kernel (tcgen05 scores)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)",
                     "traffic": traffic, "algorithmic_bytes": nbytes["indexer"],
                     "launch_us": idx_ms * 1000},
        "layer_roofline": {"algorithmic_bytes": nbytes["total"], "achieved_gbs": layer_gbs,
                           "frac": layer_gbs / peak},
        "stage_rooflines": {
            name: {"algorithmic_bytes": nbytes[key], "stage_us": stage_mean[j] * 1000,
                   "achieved_gbs": nbytes[key] / (stage_mean[j] * 1e-3) / 1e9,
                   "frac": nbytes[key] / (stage_mean[j] * 1e-3) / 1e9 / peak}
            for name, key, j in (("indexer", "indexer", 1), ("topk", "topk", 2),
                                 ("attention (+ split merge)", "attention", 3))},
        "stage_us": {"append_compress": stage_mean[0] * 1000, "indexer": stage_mean[1] * 1000,
                     "topk": stage_mean[2] * 1000, "attention": stage_mean[3] * 1000},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e * 1000 / world, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": wall,
        "topk_rows_per_s": topk,
        "multi_layer_graph": multi,
    }
    print(json.dumps(line), flush=True)


def run_profile(ctx=None):
    """Two layer steps of the bench workload (the first warms up), for ncu."""
    _lib.load(build_if_missing=True)
    shape = synth.FULL
    L, g = build_workload(0, ctx)
    B = L.numel()
    out = torch.empty(B, shape.Hq, shape.Dv, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, shape.Hq, dtype=torch.float32, device="cuda")
    desc = _lib.layer_desc(g, out, lse, torch.empty_like(g.seq_len_in),
                           torch.empty(B, shape.k, dtype=torch.int32, device="cuda"),
                           torch.empty(g.kv_pool.shape[0], dtype=torch.float32, device="cuda"))
    ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
    for _ in range(2):
        _lib.hsa_layer_decode(desc, ws=ws)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    print(json.dumps({"profile": "ok", "sum_c4_entries": int((L // 4).sum())}))


def multi_layer_graph(args, flush, nstates=4, iters=10):
    """A decode step over `args.layers` C4 layers (the bench's shapes; layer i
    works on state i mod nstates, each larger than L2) captured once in a CUDA
    graph: us per layer of the replayed step, next to the same layers launched
    one call at a time."""
    shape = synth.FULL
    states = []
    for j in range(nstates):
        L, g = build_workload(0) if j == 0 else (None, None)
        if j:
            seed = synth.SEED["c4layer"] + 7919 * j
            L = synth.c4_lengths(seed, 64)
            g = synth.filled_state(seed, 4, shape, L, device="cuda", name=f"layer{j}")
        B = L.numel()
        out = torch.empty(B, shape.Hq, shape.Dv, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, shape.Hq, dtype=torch.float32, device="cuda")
        idx = torch.empty(B, shape.k, dtype=torch.int32, device="cuda")
        scores = torch.empty(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
        desc = _lib.layer_desc(g, out, lse, torch.empty_like(g.seq_len_in), idx, scores)
        ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
        states.append((g, desc, ws, out, lse, idx, scores))
    descs = [states[i % nstates] for i in range(args.layers)]

    def eager():
        for _, desc, ws, *_ in descs:
            _lib.hsa_layer_decode(desc, ws=ws)

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
    for _, _, ws, *_ in states:
        assert _lib.hsa_workspace_status(ws) == 0
    per = {m: statistics.mean(v) * 1000 / args.layers for m, v in times.items()}
    return {"layers": args.layers, "states": nstates, "us_per_layer_graph": per["graph"],
            "us_per_layer_eager": per["eager"],
            "note": "C4 layers of the bench workload, layer i on state i mod 4; L2 flushed "
                    "before each step, not between layers"}


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


def topk_rows_per_s(flush, iters=20):
    """Standalone Lightning TopK on 64 rows x 262,144 fp32 (5% copied entries),
    k=512: rows per second, L2 flushed before each launch."""
    x = synth.topk_scores(synth.SEED["topk"], 64, 262144, 0.05, device="cuda").reshape(-1)
    offs = torch.arange(65, dtype=torch.int64, device="cuda") * 262144
    idx = torch.empty(64, 512, dtype=torch.int32, device="cuda")
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(64, x.numel(), 512))
    for _ in range(3):
        _lib.hsa_topk(x, offs, 512, idx=idx, ws=ws, with_vals=False)
    ts = []
    for i in range(iters):
        flush(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        _lib.hsa_topk(x, offs, 512, idx=idx, ws=ws, with_vals=False)
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.mean(ts)
    peak, _ = measured_peaks()
    gbs = x.numel() * 4 / (ms * 1e-3) / 1e9
    return {"value": 64 / (ms * 1e-3), "unit": "rows/s", "us_per_call": ms * 1000,
            "config": "64 x 262,144 fp32, 5% copied entries, k=512",
            "achieved_gbs": gbs, "frac_of_hbm": gbs / peak}


def indexer_traffic():
    """DRAM bytes per indexer launch from the committed ncu summary, if it was
    taken on the current indexer source (else null)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "indexer_c4layer_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for name in ("indexer.cu", "tc.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "hybrid_sparse_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


if __name__ == "__main__":
    main()
