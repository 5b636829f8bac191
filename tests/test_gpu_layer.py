"""End-to-end parity of one hybrid-layer decode step (append, compress on block
completion, indexer, top-k, attention) against the oracle's composition."""
import math

import numpy as np
import pytest
import torch

from helpers import bf16_bits, bf16_values, np_state, set_agreement
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


def rel_err(gpu, ref):
    return np.abs(gpu - ref) / np.maximum(np.abs(ref), 1e-2)


def score_tol(iq, w, keys, offs, factor):
    """factor * sum_h |w_h| sum_d |q_hd k_jd| per row (keys in pool rows)."""
    q = np.abs(bf16_values(iq))
    k = np.abs(bf16_values(keys))
    out = np.zeros(k.shape[0])
    for b in range(len(offs) - 1):
        lo, hi = int(offs[b]), int(offs[b + 1])
        out[lo:hi] = (k[lo:hi] @ q[b].T) @ np.abs(w[b].astype(np.float64))
    return factor * out


def run_gpu_step(g, out_dtype=torch.bfloat16, seq_len_out=None, max_pool_rows=None):
    B = g.seq_len_in.numel()
    sh = g.shape
    out = torch.empty(B, sh.Hq, sh.Dv, dtype=out_dtype, device="cuda")
    lse = torch.empty(B, sh.Hq, dtype=torch.float32, device="cuda")
    so = torch.empty_like(g.seq_len_in) if seq_len_out is None else seq_len_out
    res = {"out": out, "lse": lse, "seq_len_out": so}
    kw = {}
    if g.kind == 4:
        res["idx"] = torch.empty(B, sh.k, dtype=torch.int32, device="cuda")
        res["scores"] = torch.zeros(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
        kw = dict(topk_idx=res["idx"], scores=res["scores"])
    desc = _lib.layer_desc(g, out, lse, so, max_pool_rows=max_pool_rows, **kw)
    ws = _lib.hsa_layer_decode(desc)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    return res


def build_tiny(kind, L=4096, slack=1):
    """Tiny layer from raw tokens: the oracle and the GPU each compress the
    history into their own pools."""
    st, raw = synth.raw_token_state(synth.SEED["tiny"], kind, synth.TINY, L, slack=slack)
    return st, raw


def gpu_prefix_pools(g, raw, kind):
    kv = _lib.hsa_compress(raw["kv"].cuda(), raw["z"].cuda(), g.b_kv, kind)
    g.kv_pool[:kv.shape[1]] = kv[0]
    if kind == 4:
        ks = _lib.hsa_compress(raw["ik"].cuda(), raw["iz"].cuda(), g.b_ik, 4)
        g.key_pool[:ks.shape[1]] = ks[0]


def oracle_prefix_pools(oracle_mod, s, raw, kind):
    pre = oracle_mod.compress(bf16_bits(raw["kv"]), bf16_bits(raw["z"]), s["b_kv"], kind)[0]
    s["kv_pool"][:pre.shape[0]] = oracle_mod.float_to_bf16(pre.astype(np.float32))
    if kind == 4:
        pk = oracle_mod.compress(bf16_bits(raw["ik"]), bf16_bits(raw["iz"]), s["b_ik"], 4)[0]
        s["key_pool"][:pk.shape[0]] = oracle_mod.float_to_bf16(pk.astype(np.float32))


def check_step(oracle_mod, g, s, res, ref, min_agree):
    kind = g.kind
    L = ref["seq_len_out"].astype(np.int64)
    assert np.array_equal(res["seq_len_out"].cpu().numpy(), ref["seq_len_out"])
    offs = s["pool_offsets"]
    counts = L // kind
    # pools: every live row within the compressor tolerance
    gp = bf16_values(bf16_bits(g.kv_pool.cpu()))
    rp = bf16_values(s["kv_pool"])
    for b in range(len(L)):
        lo = int(offs[b])
        n = int(counts[b])
        if n:
            assert rel_err(gp[lo:lo + n], rp[lo:lo + n]).max() <= 5e-3
    assert np.array_equal(bf16_bits(g.swa.cpu()), s["swa"])
    idx_used = None
    if kind == 4:
        gs = res["scores"].cpu().numpy().astype(np.float64)
        key_rows, key_offs = oracle_mod.compact(s["key_pool"], offs, counts)
        gsc = np.concatenate([gs[int(offs[b]):int(offs[b]) + int(counts[b])] for b in range(len(L))])
        # keys may differ by one bf16 rounding step: |dk| <= 2^-8 |k|
        tol = score_tol(s["iq"], s["w"], key_rows, key_offs, 2.0 ** -7) + 1e-30
        assert np.all(np.abs(gsc - ref["scores64"]) <= tol)
        gidx = res["idx"].cpu().numpy()
        # top-k bit-exact on the GPU's own fp32 scores
        own, _ = oracle_mod.topk(gsc.astype(np.float32), key_offs, s["k"], threads=16)
        assert np.array_equal(gidx, own)
        agree = set_agreement(gidx, ref["idx"], counts, s["k"])
        assert agree >= min_agree, f"top-k set agreement {agree:.5f}"
        idx_used = gidx
    # attention: oracle fed the GPU's selected indices (its own pools)
    kv_rows, kv_offs = oracle_mod.compact(s["kv_pool"], offs, counts)
    o_ref, l_ref = oracle_mod.decode_attn(s["q"], s["swa"], L.astype(np.int32), s["swa"].shape[1],
                                          kv_rows, kv_offs, idx_used, s["scale"], s["Dv"],
                                          threads=16)
    go = res["out"].float().cpu().numpy()
    err = np.abs(go - o_ref).max()
    assert err <= 1e-2, f"attention max abs err {err:.3e}"
    lerr = np.abs(res["lse"].cpu().numpy() - l_ref).max()
    assert lerr <= 2.0 ** -8
    return err


@pytest.mark.parametrize("kind", [4, 128])
def test_layer_tiny_from_raw_tokens(oracle_mod, kind):
    st, raw = build_tiny(kind)
    s = np_state(st)
    oracle_prefix_pools(oracle_mod, s, raw, kind)
    g = st.to("cuda")
    gpu_prefix_pools(g, raw, kind)
    res = run_gpu_step(g)
    ref = oracle_mod.layer_decode(s)
    # one sequence with 64 of 1,024 entries: allow one flip at the threshold
    check_step(oracle_mod, g, s, res, ref, min_agree=62 / 64)


def test_layer_tiny_dense_equivalence_k_covers_all():
    """k >= the number of C4 entries: the sparse C4 layer equals dense attention
    over every entry (plus the window)."""
    shape = synth.LayerShape(Hq=8, Dqk=128, Dv=128, Hi=2, Di=32, k=1024, W=64)
    st, raw = synth.raw_token_state(synth.SEED["tiny"], 4, shape, 4096)
    g = st.to("cuda")
    gpu_prefix_pools(g, raw, 4)
    res = run_gpu_step(g, out_dtype=torch.float32)
    # dense attention over the same pool rows and window
    n = 4096 // 4
    o, l = _lib.hsa_decode_attn(g.q, g.swa, res["seq_len_out"], g.kv_pool[:n].contiguous(),
                                torch.tensor([0, n], dtype=torch.int64, device="cuda"), None,
                                max_extra_rows=n, scale=shape.scale, Dv=128,
                                out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (res["out"] - o).abs().max().item() <= 1e-3
    assert (res["lse"] - l).abs().max().item() <= 1e-3


@pytest.mark.parametrize("kind", [4, 128])
def test_layer_multi_step_in_place(oracle_mod, kind):
    """Six consecutive in-place steps (seq_len_out aliases seq_len_in) crossing
    block completions (C4: two; C128: one, at L = 4096); the state carried by
    the rings stays in parity.  With aliased lengths the C128 attention waits
    for the append before reading any length (with separate ones it starts
    while the append runs)."""
    st, raw = build_tiny(kind, L=4091, slack=4)   # room for the blocks of 6 more tokens
    s = np_state(st)
    oracle_prefix_pools(oracle_mod, s, raw, kind)
    g = st.to("cuda")
    gpu_prefix_pools(g, raw, kind)
    for step in range(6):
        name = f"step{step}"
        for key in ("kv_new", "z_new") + (("ik_new", "iz_new") if kind == 4 else ()):
            v = synth.normal_bf16(synth.SEED["tiny"], f"{name}.{key}", tuple(getattr(st, key).shape))
            getattr(g, key).copy_(v.cuda())
            s[key] = bf16_bits(v)
        res = run_gpu_step(g, seq_len_out=g.seq_len_in)
        ref = oracle_mod.layer_decode(s)
        s["seq_len_in"] = ref["seq_len_out"].copy()
        assert int(g.seq_len_in.item()) == 4091 + step
        check_step(oracle_mod, g, s, res, ref, min_agree=62 / 64)


def test_layer_step_is_idempotent_with_separate_output_length():
    L = synth.c4_lengths(synth.SEED["c4layer"], 8, 4000, 9000)
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda", name="idem")
    a = run_gpu_step(g)
    b = run_gpu_step(g)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["idx"], b["idx"])
    assert torch.equal(a["seq_len_out"], L.cuda())


def test_layer_attention_waits_for_q_ready_event():
    """q arrives on a side stream after a delay; the layer waits for the event
    right before the attention (the only reader of q), so the upload overlaps
    the append, indexer and top-k, and the result equals the step with q
    resident beforehand."""
    L = synth.c4_lengths(synth.SEED["c4layer"], 8, 4000, 9000)
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda", name="qev")
    ref = run_gpu_step(g)
    q_host = g.q.cpu().pin_memory()
    g.q.zero_()
    B, sh = L.numel(), g.shape
    out = torch.empty(B, sh.Hq, sh.Dv, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sh.Hq, dtype=torch.float32, device="cuda")
    so = torch.empty_like(g.seq_len_in)
    idx = torch.empty(B, sh.k, dtype=torch.int32, device="cuda")
    scores = torch.zeros(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    ready = torch.cuda.Event()
    ready.record(side)                    # the event exists before its handle is taken
    desc = _lib.layer_desc(g, out, lse, so, topk_idx=idx, scores=scores,
                           q_ready_event=ready.cuda_event)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(2_000_000)      # about a millisecond: q lands after the top-k
        g.q.copy_(q_host, non_blocking=True)
        ready.record(side)
    ws = _lib.hsa_layer_decode(desc)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    assert torch.equal(out, ref["out"]) and torch.equal(lse, ref["lse"])
    assert torch.equal(idx, ref["idx"])


def test_layer_c4_full_128k_batch64(oracle_mod):
    """The headline workload: batch 64, contexts U[16384, 131072], 64 heads x
    576, indexer 8 x 128, top-512, window 128; every stage against the oracle."""
    L = synth.c4_lengths(synth.SEED["c4layer"], 64)
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda")
    s = np_state(g)           # snapshot before the GPU step mutates rings and pools
    res = run_gpu_step(g)
    ref = oracle_mod.layer_decode(s, threads=16)
    check_step(oracle_mod, g, s, res, ref, min_agree=0.999)


@pytest.mark.parametrize("kind", [4, 128])
def test_layer_long_context_batch4(oracle_mod, kind):
    """The 1M-token pair: batch 4 at L = 1,048,576 (this step completes a block
    for both ratios), C4 top-512 over 262,144 entries or C128 dense over 8,192."""
    L = torch.full((4,), 1048576, dtype=torch.int32)
    g = synth.filled_state(synth.SEED["longctx"], kind, synth.FULL, L, device="cuda",
                           name=f"long{kind}")
    s = np_state(g)
    res = run_gpu_step(g)
    ref = oracle_mod.layer_decode(s, threads=16)
    check_step(oracle_mod, g, s, res, ref, min_agree=0.999)


@pytest.mark.parametrize("B", [8, 64])
@pytest.mark.parametrize("pattern", ["all_equal", "few_distinct", "negative_w"])
def test_layer_topk_ties_through_the_indexer_histogram(oracle_mod, pattern, B):
    """Tie-heavy score patterns through the layer's top-k: at B = 8 the
    standalone top-k kernels, at B = 64 the selection fused into the attention
    kernel, which starts from the per-row key histogram the indexer builds.
    All scores equal (a threshold bin larger than shared memory: radix select
    over the workspace), keys repeating a few distinct rows (many equal scores
    in the threshold bin, ordered by index), negative head weights (scores
    <= 0, -0.0 equal to +0.0).  Each step runs twice: the histogram is zeroed
    again after use, so the second step must give the same, bit-exact result."""
    L = synth.c4_lengths(synth.SEED["c4layer"], B, 4000, 131072)
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda",
                           name=f"tie{pattern}{B}")
    if pattern == "all_equal":
        g.iq.zero_()
    elif pattern == "few_distinct":
        offs = g.pool_offsets.cpu()
        for b in range(L.numel()):
            lo, hi = int(offs[b]), int(offs[b + 1])
            src = synth.randint(synth.SEED["c4layer"], f"tie.src.{b}", hi - lo, 0, 149)
            g.key_pool[lo:hi] = g.key_pool[lo + src.cuda()].clone()
    else:
        g.w.neg_()
    counts = (L.to(torch.int64) // 4).numpy()
    offs = g.pool_offsets.cpu().numpy()
    key_offs = np.zeros(len(counts) + 1, np.int64)
    key_offs[1:] = np.cumsum(counts)
    first = None
    for _ in range(2):
        res = run_gpu_step(g)
        gs = res["scores"].cpu().numpy()
        gsc = np.concatenate([gs[int(offs[b]):int(offs[b]) + int(counts[b])]
                              for b in range(len(counts))])
        own, _ = oracle_mod.topk(gsc.astype(np.float32), key_offs, g.shape.k, threads=16)
        gidx = res["idx"].cpu().numpy()
        assert np.array_equal(gidx, own)
        if first is None:
            first = gidx
        assert np.array_equal(gidx, first)
    if pattern == "all_equal":
        assert np.all(gsc == 0)
        assert np.array_equal(first[:, :16], np.tile(np.arange(16, dtype=np.int32), (B, 1)))


def _fused_case_lengths(B, tag):
    """Ragged context lengths: mostly U[64, 131072], plus short windows (L < 128)
    and rows shorter than k = 512 (L < 2048)."""
    L = synth.c4_lengths(synth.SEED["c4layer"], B, 64, 131072)
    special = [1, 3, 64, 127, 128, 129, 1000, 2047, 2048, 2052, 4096, 131072]
    for i, v in enumerate(special[:B]):
        L[(7 * i + len(tag)) % B] = v
    return L


@pytest.mark.parametrize("B", [50, 76, 100])
def test_layer_fused_selection_matches_separate_kernels(oracle_mod, B):
    """The layer's selection fused into the attention kernel (splits per token:
    3, 2, 1 at these batches) gives the same top-k list, bit for bit, as the
    same step with the top-k in its own kernels (a pool-row bound above
    32,768 selects that path), and the oracle's top-k of the GPU's scores; the
    outputs agree to fp32 summation order (the fused kernel attends the
    selected rows in a fixed order that is not the sorted one).  Some
    sequences repeat a few distinct keys (ties in the threshold bin)."""
    L = _fused_case_lengths(B, f"f{B}")
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda", name=f"fused{B}")
    offs_t = g.pool_offsets.cpu()
    for b in range(0, B, 5):
        lo, hi = int(offs_t[b]), int(offs_t[b + 1])
        src = synth.randint(synth.SEED["c4layer"], f"fused.src.{b}", hi - lo, 0, 99)
        g.key_pool[lo:hi] = g.key_pool[lo + src.cuda()].clone()
    s = np_state(g) if B == 76 else None
    sep = run_gpu_step(g, max_pool_rows=40000)
    fused = run_gpu_step(g)
    assert torch.equal(sep["idx"], fused["idx"])
    # bf16 outputs: one rounding step at most; lse: fp32 summation order
    assert torch.allclose(sep["out"].float(), fused["out"].float(), rtol=2.0 ** -7, atol=1e-5)
    assert torch.allclose(sep["lse"], fused["lse"], rtol=0, atol=1e-4)
    # the same step again: the fused path is deterministic
    again = run_gpu_step(g)
    assert torch.equal(again["out"], fused["out"]) and torch.equal(again["idx"], fused["idx"])
    counts = (L.to(torch.int64) // 4).numpy()
    offs = offs_t.numpy()
    key_offs = np.zeros(B + 1, np.int64)
    key_offs[1:] = np.cumsum(counts)
    gs = fused["scores"].cpu().numpy()
    gsc = np.concatenate([gs[int(offs[b]):int(offs[b]) + int(counts[b])] for b in range(B)])
    own, _ = oracle_mod.topk(gsc.astype(np.float32), key_offs, g.shape.k, threads=16)
    assert np.array_equal(fused["idx"].cpu().numpy(), own)
    if s is not None:   # one batch also against the oracle's whole step
        ref = oracle_mod.layer_decode(s, threads=16)
        check_step(oracle_mod, g, s, fused, ref, min_agree=0.999)
