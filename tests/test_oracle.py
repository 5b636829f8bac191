"""Pins for the CPU oracle: each stage checked against something other than itself
(hand-worked closed forms, special cases that reduce to a library routine,
invariants, brute force on tiny inputs).  CPU only."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from helpers import bf16_bits, bf16_values, closed_form, golden
from hybrid_sparse_attention_gb300 import synth

RNG_SEED = 0x5EED


def _normal_bits(name, shape, std=1.0):
    return bf16_bits(synth.normal_bf16(RNG_SEED, name, shape, std))


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_bit_patterns(oracle_mod):
    # values chosen on the binary32 grid around bf16 rounding boundaries
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,                 # exact tie, even kept
        1.0 + 3 * 2.0 ** -8: 0x3F82,             # exact tie, rounds up to even
        1.0 + 2.0 ** -8 + 2.0 ** -20: 0x3F81,    # just above the tie
        -2.5: 0xC020,
        float("inf"): 0x7F80,
        float("-inf"): 0xFF80,
        3.3895313892515355e38: 0x7F7F,           # largest finite bf16
        3.4028234663852886e38: 0x7F80,           # FLT_MAX rounds to +inf
        1e-45: 0x0000,                           # smallest subnormal rounds to zero
        -0.0: 0x8000,
    }
    x = np.array(list(cases.keys()), np.float32)
    got = oracle_mod.float_to_bf16(x)
    assert [int(v) for v in got] == list(cases.values())
    nan = oracle_mod.float_to_bf16(np.array([np.nan], np.float32))
    assert (int(nan[0]) & 0x7F80) == 0x7F80 and (int(nan[0]) & 0x7F) != 0


def test_bf16_rounding_matches_torch(oracle_mod):
    x = synth.normal(RNG_SEED, "bf16.rt", (20000,), std=3.0).numpy()
    assert np.array_equal(oracle_mod.float_to_bf16(x), bf16_bits(torch.from_numpy(x)))
    bits = np.arange(0, 65536, dtype=np.uint16)
    finite = (bits & 0x7F80) != 0x7F80
    assert np.array_equal(oracle_mod.bf16_to_double(bits)[finite], bf16_values(bits)[finite])


# ---------------------------------------------------------------- compressor

def test_compress_worked_example(oracle_mod):
    g = golden("compress_worked.json")
    kv = bf16_bits(np.array(g["kv"])[None])
    z = bf16_bits(np.array(g["z"])[None])
    b = np.array(g["b"], np.float32)
    got = oracle_mod.compress(kv, z, b, g["r"])[0, 0]
    want = [closed_form(e) for e in g["expected"]]
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)


def test_compress_ratio_one_is_identity(oracle_mod):
    kv = _normal_bits("c.kv1", (2, 16, 8))
    z = _normal_bits("c.z1", (2, 16, 8))
    b = synth.normal(RNG_SEED, "c.b1", (1, 8)).numpy()
    got = oracle_mod.compress(kv, z, b, 1)
    assert np.array_equal(got, bf16_values(kv))


def test_compress_constant_gate_is_block_mean(oracle_mod):
    kv = _normal_bits("c.kv2", (2, 32, 5))
    z = np.broadcast_to(bf16_bits(np.float32(0.75)), kv.shape).copy()
    b = np.full((4, 5), -1.25, np.float32)
    got = oracle_mod.compress(kv, z, b, 4)
    want = bf16_values(kv).reshape(2, 8, 4, 5).mean(axis=2)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)


def test_compress_dominant_logit_selects_row(oracle_mod):
    kv = _normal_bits("c.kv3", (1, 8, 6))
    z = np.zeros((1, 8, 6), np.uint16)
    z[0, 1::4] = bf16_bits(np.float32(40.0))  # position 1 of every block dominates
    b = np.zeros((4, 6), np.float32)
    got = oracle_mod.compress(kv, z, b, 4)
    np.testing.assert_allclose(got[0], bf16_values(kv)[0, 1::4], rtol=0, atol=1e-15)


def test_compress_library_softmax_and_invariants(oracle_mod):
    S, T, C, r = 2, 64, 12, 4
    kv = _normal_bits("c.kv4", (S, T, C))
    z = _normal_bits("c.z4", (S, T, C))
    b = (np.round(synth.normal(RNG_SEED, "c.b4", (r, C), 0.5).numpy() * 64) / 64).astype(np.float32)
    got = oracle_mod.compress(kv, z, b, r)
    # scipy softmax over the block positions (a library routine)
    logits = bf16_values(z).reshape(S, T // r, r, C) + b[None, None].astype(np.float64)
    wts = scipy.special.softmax(logits, axis=2)
    want = (wts * bf16_values(kv).reshape(S, T // r, r, C)).sum(axis=2)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
    # convex combination: inside [min, max] of the block per channel
    blk = bf16_values(kv).reshape(S, T // r, r, C)
    assert np.all(got >= blk.min(axis=2) - 1e-12) and np.all(got <= blk.max(axis=2) + 1e-12)
    # shift invariance: a per-channel constant added to b (exact in fp32) changes nothing
    got_shift = oracle_mod.compress(kv, z, b + np.float32(3.0), r)
    np.testing.assert_allclose(got_shift, got, rtol=1e-12, atol=1e-14)
    # linearity in kv: doubling (exact in bf16) doubles the output
    kv2 = bf16_bits(2.0 * bf16_values(kv).astype(np.float32))
    np.testing.assert_allclose(oracle_mod.compress(kv2, z, b, r), 2 * got, rtol=1e-14, atol=0)


def test_compress_additivity_small_integers(oracle_mod):
    # kv with small integer values so the sum of two inputs stays exact in bf16
    a = (np.arange(2 * 16 * 3).reshape(2, 16, 3) % 7 - 3).astype(np.float32)
    c = (np.arange(2 * 16 * 3).reshape(2, 16, 3) % 5 - 2).astype(np.float32)
    z = _normal_bits("c.z5", (2, 16, 3))
    b = np.zeros((4, 3), np.float32)
    ya = oracle_mod.compress(bf16_bits(a), z, b, 4)
    yc = oracle_mod.compress(bf16_bits(c), z, b, 4)
    yac = oracle_mod.compress(bf16_bits(a + c), z, b, 4)
    np.testing.assert_allclose(yac, ya + yc, rtol=1e-13, atol=1e-13)


def test_compress_drops_trailing_partial_block(oracle_mod):
    kv = _normal_bits("c.kv6", (1, 10, 4))
    z = _normal_bits("c.z6", (1, 10, 4))
    b = np.zeros((4, 4), np.float32)
    full = oracle_mod.compress(kv, z, b, 4)
    assert full.shape == (1, 2, 4)
    np.testing.assert_array_equal(full, oracle_mod.compress(kv[:, :8], z[:, :8], b, 4))


# ---------------------------------------------------------------- indexer

def test_indexer_worked_example(oracle_mod):
    g = golden("indexer_worked.json")
    q = bf16_bits(np.array(g["q"])[None])
    w = np.array([g["w"]], np.float32)
    keys = bf16_bits(np.array(g["keys"]))
    got = oracle_mod.indexer_scores(q, w, keys, np.array([0, 4], np.int64))
    np.testing.assert_array_equal(got, g["expected"])


def test_indexer_one_hot_reduces_to_relu_of_a_key_column(oracle_mod):
    B, Hi, Di, n = 2, 3, 16, 50
    keys = _normal_bits("i.k1", (B * n, Di))
    q = np.zeros((B, Hi, Di), np.float32)
    q[0, 1, 5] = 1.0
    q[1, 2, 11] = 1.0
    w = np.zeros((B, Hi), np.float32)
    w[0, 1] = 0.5
    w[1, 2] = 0.25
    offs = np.array([0, n, 2 * n], np.int64)
    got = oracle_mod.indexer_scores(bf16_bits(q), w, keys, offs)
    kv = bf16_values(keys)
    np.testing.assert_array_equal(got[:n], 0.5 * np.maximum(0.0, kv[:n, 5]))
    np.testing.assert_array_equal(got[n:], 0.25 * np.maximum(0.0, kv[n:, 11]))


def test_indexer_library_matmul_linearity_nonnegativity(oracle_mod):
    B, Hi, Di = 3, 4, 32
    counts = [17, 0, 40]
    offs = np.zeros(B + 1, np.int64)
    offs[1:] = np.cumsum(counts)
    keys = _normal_bits("i.k2", (int(offs[-1]), Di))
    q = _normal_bits("i.q2", (B, Hi, Di))
    w1 = synth.uniform(RNG_SEED, "i.w1", (B, Hi)).numpy()
    w2 = synth.uniform(RNG_SEED, "i.w2", (B, Hi)).numpy()
    got = oracle_mod.indexer_scores(q, w1, keys, offs)
    assert np.all(got >= 0)
    kf, qf = bf16_values(keys), bf16_values(q)
    for b in range(B):
        lo, hi = offs[b], offs[b + 1]
        want = np.maximum(kf[lo:hi] @ qf[b].T, 0.0) @ w1[b].astype(np.float64)
        np.testing.assert_allclose(got[lo:hi], want, rtol=1e-12, atol=1e-12)
    g2 = oracle_mod.indexer_scores(q, w2, keys, offs)
    g12 = oracle_mod.indexer_scores(q, (w1.astype(np.float64) + w2).astype(np.float32), keys, offs)
    np.testing.assert_allclose(g12, got + g2, rtol=1e-6, atol=1e-9)  # w1+w2 rounds to fp32


# ---------------------------------------------------------------- top-k

def _topk_rows(rows):
    vals = np.concatenate([np.array([float(v) for v in r], np.float32) for r in rows]) \
        if any(len(r) for r in rows) else np.zeros(0, np.float32)
    offs = np.zeros(len(rows) + 1, np.int64)
    offs[1:] = np.cumsum([len(r) for r in rows])
    return vals, offs


def test_topk_worked_example(oracle_mod):
    g = golden("topk_worked.json")
    vals, offs = _topk_rows(g["rows"])
    for case in g["cases"]:
        idx, _ = oracle_mod.topk(vals, offs, case["k"])
        assert idx.tolist() == case["expected"]


def _lexsort_reference(row, k):
    order = np.lexsort((np.arange(row.size), -row.astype(np.float64)))  # value desc, index asc
    out = np.full(k, -1, np.int32)
    m = min(k, row.size)
    out[:m] = order[:m]
    return out


def test_topk_matches_library_sort_on_tied_rows(oracle_mod):
    rows = [synth.topk_scores(RNG_SEED, 1, n, 0.05)[0].numpy() for n in (1, 7, 600, 5000, 33000)]
    rows.append(synth.pair_ties_at_top(torch.from_numpy(rows[-1]), 600).numpy())
    rows.append(np.round(rows[3] * 4) / 4)  # heavy duplicates
    vals = np.concatenate(rows).astype(np.float32)
    offs = np.zeros(len(rows) + 1, np.int64)
    offs[1:] = np.cumsum([r.size for r in rows])
    for k in (1, 64, 512):
        idx, v = oracle_mod.topk(vals, offs, k)
        for i, r in enumerate(rows):
            assert np.array_equal(idx[i], _lexsort_reference(r, k))
            m = min(k, r.size)
            assert np.array_equal(v[i, :m], r[idx[i, :m]])
            if r.size >= k:   # k-th value equals numpy's partition (nth_element)
                assert v[i, k - 1] == np.partition(r, r.size - k)[r.size - k]


def test_topk_special_rows(oracle_mod):
    n, k = 1000, 64
    equal = np.full(n, 0.5, np.float32)
    rev = np.arange(n, dtype=np.float32)[::-1].copy()
    zeros = np.where(np.arange(n) % 2 == 0, -0.0, 0.0).astype(np.float32)
    infs = np.full(n, -np.inf, np.float32)
    infs[[3, 500, 999]] = np.inf
    vals = np.concatenate([equal, rev, zeros, infs])
    offs = np.arange(5, dtype=np.int64) * n
    idx, v = oracle_mod.topk(vals, offs, k)
    assert idx[0].tolist() == list(range(k))
    assert idx[1].tolist() == list(range(k))
    assert idx[2].tolist() == list(range(k))          # -0.0 == +0.0: index order
    assert idx[3].tolist() == [3, 500, 999] + [i for i in range(n) if i not in (3, 500, 999)][:k - 3]
    big, _ = oracle_mod.topk(rev[:10], np.array([0, 10], np.int64), 16)
    assert big[0].tolist() == list(range(10)) + [-1] * 6


def test_topk_rejects_nan(oracle_mod):
    vals = np.array([1.0, np.nan, 2.0], np.float32)
    with pytest.raises(ValueError):
        oracle_mod.topk(vals, np.array([0, 3], np.int64), 2)


# ---------------------------------------------------------------- attention

def _attn_case(g, use_idx):
    q = bf16_bits(np.array(g["q"])[None, None])
    swa = bf16_bits(np.array(g["swa"])[None])
    extra = bf16_bits(np.array(g["extra"]))
    offs = np.array([0, len(g["extra"])], np.int64)
    idx = np.array([g["idx"]], np.int32) if use_idx else None
    return q, swa, extra, offs, idx


def test_attention_worked_example(oracle_mod):
    g = golden("attn_worked.json")
    for use_idx, key in ((True, "expected_sparse"), (False, "expected_dense")):
        q, swa, extra, offs, idx = _attn_case(g, use_idx)
        o, lse = oracle_mod.decode_attn(q, swa, np.array([g["seq_len"]], np.int32), swa.shape[1],
                                        extra, offs, idx, 1.0, g["Dv"])
        np.testing.assert_allclose(o[0, 0], [closed_form(e) for e in g[key]["out"]], rtol=1e-14)
        assert math.isclose(lse[0, 0], closed_form(g[key]["lse"]), rel_tol=1e-14)


def _rand_attn(B=3, Hq=4, D=16, Dv=12, W=8, n=(5, 0, 30), L=(3, 20, 8), k=6):
    offs = np.zeros(B + 1, np.int64)
    offs[1:] = np.cumsum(n)
    q = _normal_bits("a.q", (B, Hq, D))
    swa = _normal_bits("a.swa", (B, W, D))
    extra = _normal_bits("a.extra", (int(offs[-1]), D))
    idx = np.full((B, k), -1, np.int32)
    for b in range(B):
        m = min(k, n[b])
        idx[b, :m] = (np.arange(m) * 7 + b) % max(n[b], 1)
    return q, swa, np.array(L, np.int32), W, extra, offs, idx, Dv


def test_attention_matches_library_sdpa(oracle_mod):
    q, swa, L, W, extra, offs, idx, Dv = _rand_attn()
    scale = 0.37
    o, lse = oracle_mod.decode_attn(q, swa, L, W, extra, offs, idx, scale, Dv)
    qf, sf, ef = bf16_values(q), bf16_values(swa), bf16_values(extra)
    for b in range(q.shape[0]):
        rows = [sf[b, p % W] for p in range(max(0, L[b] - W), L[b])]
        rows += [ef[offs[b] + j] for j in idx[b] if j >= 0]
        K = torch.tensor(np.array(rows))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(qf[b])[None], K[None], K[None, :, :Dv], scale=scale)[0]
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=1e-12, atol=1e-13)
        want_lse = torch.logsumexp(scale * torch.tensor(qf[b]) @ K.T, dim=1).numpy()
        np.testing.assert_allclose(lse[b], want_lse, rtol=1e-13)


def test_attention_single_row_and_equal_logits(oracle_mod):
    q, swa, L, W, extra, offs, idx, Dv = _rand_attn()
    # one window row, nothing compressed: o = that row's value part, lse = its logit
    o, lse = oracle_mod.decode_attn(q, swa, np.array([1, 1, 1], np.int32), W, None, None, None,
                                    1.0, Dv)
    for b in range(3):
        assert np.array_equal(o[b], np.broadcast_to(bf16_values(swa)[b, 0, :Dv], o[b].shape))
    # q = 0: all logits equal -> mean of the values, lse = log(count)
    zq = np.zeros_like(q)
    o, lse = oracle_mod.decode_attn(zq, swa, L, W, extra, offs, None, 1.0, Dv)
    for b in range(3):
        rows = [bf16_values(swa)[b, p % W] for p in range(max(0, L[b] - W), L[b])]
        rows += list(bf16_values(extra)[offs[b]:offs[b + 1]])
        np.testing.assert_allclose(o[b, 0], np.mean(rows, axis=0)[:Dv], rtol=1e-13, atol=1e-15)
        assert math.isclose(lse[b, 0], math.log(len(rows)), rel_tol=1e-14)


def test_attention_split_and_lse_combine_equals_whole(oracle_mod):
    q, swa, L, W, extra, offs, idx, Dv = _rand_attn()
    o, lse = oracle_mod.decode_attn(q, swa, L, W, extra, offs, idx, 0.5, Dv)
    o1, l1 = oracle_mod.decode_attn(q, swa, L, W, None, None, None, 0.5, Dv)       # window only
    o2, l2 = oracle_mod.decode_attn(q, swa, np.zeros(3, np.int32), W, extra, offs, idx, 0.5, Dv)
    m = np.maximum(l1, l2)
    a1, a2 = np.exp(l1 - m), np.exp(np.where(np.isinf(l2), -np.inf, l2 - m))
    comb = (a1[..., None] * o1 + a2[..., None] * o2) / (a1 + a2)[..., None]
    np.testing.assert_allclose(comb, o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(m + np.log(a1 + a2), lse, rtol=1e-13)


def test_attention_all_indices_equals_dense(oracle_mod):
    q, swa, L, W, extra, offs, _, Dv = _rand_attn()
    n = np.diff(offs)
    k = int(n.max()) + 3
    idx = np.full((3, k), -1, np.int32)
    for b in range(3):
        idx[b, :n[b]] = np.arange(n[b])[::-1]      # any order
    o_s, l_s = oracle_mod.decode_attn(q, swa, L, W, extra, offs, idx, 0.3, Dv)
    o_d, l_d = oracle_mod.decode_attn(q, swa, L, W, extra, offs, None, 0.3, Dv)
    np.testing.assert_allclose(o_s, o_d, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(l_s, l_d, rtol=1e-14)


def test_attention_empty_set_and_bad_index(oracle_mod):
    q, swa, L, W, extra, offs, idx, Dv = _rand_attn()
    o, lse = oracle_mod.decode_attn(q, swa, np.zeros(3, np.int32), W, None, None, None, 1.0, Dv)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    bad = idx.copy()
    bad[0, 0] = 5  # sequence 0 has 5 entries: 5 is out of range
    with pytest.raises(ValueError):
        oracle_mod.decode_attn(q, swa, L, W, extra, offs, bad, 1.0, Dv)


# ---------------------------------------------------------------- layer composition

def _np_state(st):
    out = {k: (bf16_bits(v) if v.dtype == torch.bfloat16 else v.numpy().copy())
           for k, v in st.tensors().items()}
    out.update(kind=st.kind, ratio=st.ratio, Dv=st.shape.Dv, k=st.shape.k, scale=st.shape.scale)
    return out


@pytest.mark.parametrize("kind", [4, 128])
def test_layer_step_pools_match_bulk_compression_of_history(oracle_mod, kind):
    """After one decode step, the incrementally maintained pool equals the bulk
    compression of the whole token history (history + the new token)."""
    shape = synth.TINY
    L = 2 * kind if kind == 128 else 64        # the step completes a block
    st, raw = synth.raw_token_state(RNG_SEED, kind, shape, L)
    s = _np_state(st)
    kvh = bf16_bits(raw["kv"])
    zh = bf16_bits(raw["z"])
    prefix = oracle_mod.compress(kvh, zh, s["b_kv"], kind)[0]
    s["kv_pool"][:prefix.shape[0]] = oracle_mod.float_to_bf16(prefix.astype(np.float32))
    if kind == 4:
        pk = oracle_mod.compress(bf16_bits(raw["ik"]), bf16_bits(raw["iz"]), s["b_ik"], 4)[0]
        s["key_pool"][:pk.shape[0]] = oracle_mod.float_to_bf16(pk.astype(np.float32))
    res = oracle_mod.layer_decode(s)
    assert res["seq_len_out"].tolist() == [L]
    full_kv = np.concatenate([kvh[0], s["kv_new"]], axis=0)[None]
    full_z = np.concatenate([zh[0], s["z_new"]], axis=0)[None]
    bulk = oracle_mod.float_to_bf16(oracle_mod.compress(full_kv, full_z, s["b_kv"], kind)
                                    .astype(np.float32))[0]
    n = L // kind
    assert np.array_equal(s["kv_pool"][:n], bulk)
    # the SWA window now ends with the new token
    assert np.array_equal(s["swa"][0, (L - 1) % shape.W], s["kv_new"][0])
    if kind == 4:
        assert res["idx"].shape == (1, shape.k)
        assert sorted(res["idx"][0][res["idx"][0] >= 0].tolist()) == \
            sorted(set(res["idx"][0][res["idx"][0] >= 0].tolist()))


# ---------------------------------------------------------------- threading

def test_threaded_stages_equal_single_thread(oracle_mod):
    """The oracle shares out independent outputs (indexer entries, attention
    (sequence, head) pairs, top-k rows) among threads; every output is still
    computed by one thread in the same order, so any thread count gives the
    same bits as one thread."""
    B, Hi, Di = 3, 4, 32
    counts = [17, 0, 40]
    offs = np.zeros(B + 1, np.int64)
    offs[1:] = np.cumsum(counts)
    keys = _normal_bits("t.k", (int(offs[-1]), Di))
    q = _normal_bits("t.q", (B, Hi, Di))
    w = synth.uniform(RNG_SEED, "t.w", (B, Hi)).numpy()
    one = oracle_mod.indexer_scores(q, w, keys, offs, threads=1)
    for t in (2, 5, 64):
        assert np.array_equal(oracle_mod.indexer_scores(q, w, keys, offs, threads=t), one)
    ti, tv = oracle_mod.topk(one.astype(np.float32), offs, 8, threads=1)
    ti5, tv5 = oracle_mod.topk(one.astype(np.float32), offs, 8, threads=5)
    assert np.array_equal(ti, ti5) and np.array_equal(tv, tv5)
    qa, swa, L, W, extra, aoffs, idx, Dv = _rand_attn()
    o1, l1 = oracle_mod.decode_attn(qa, swa, L, W, extra, aoffs, idx, 0.3, Dv, threads=1)
    for t in (3, 16):
        o, l = oracle_mod.decode_attn(qa, swa, L, W, extra, aoffs, idx, 0.3, Dv, threads=t)
        assert np.array_equal(o, o1) and np.array_equal(l, l1)


# ---------------------------------------------------------------- FP8 E4M3 (indexer-key pool)

def test_e4m3_decode_every_code_matches_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.e4m3_to_double(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(lib))
    assert np.isnan(got).sum() == 2                          # 0x7f and 0xff
    live = ~np.isnan(got)
    assert np.array_equal(got[live], lib[live])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert got[0x38] == 1.0 and got[0xB8] == -1.0


def test_e4m3_encode_named_values(oracle_mod):
    g = golden("e4m3_worked.json")
    x = np.array([closed_form(e) for e, _, _ in g["encode"]], np.float32)
    want = [c for _, c, _ in g["encode"]]
    assert [int(v) for v in oracle_mod.float_to_e4m3(x)] == want
    assert int(oracle_mod.float_to_e4m3(np.array([np.nan], np.float32))[0]) & 0x7F == 0x7F


def test_e4m3_encode_matches_torch_rounding(oracle_mod):
    rng = np.random.default_rng(RNG_SEED)
    vals = oracle_mod.e4m3_to_double(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2                         # every tie, exactly
    x = np.concatenate([
        rng.uniform(-448, 448, 200_000),
        rng.standard_normal(100_000) * 0.02,                  # the subnormal range
        mids, -mids,
        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.float_to_e4m3(x), lib)


def test_e4m3_quantize_rows(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 1)
    x = (rng.standard_normal((300, 128)) * rng.uniform(1e-3, 50, (300, 1))).astype(np.float32)
    x[7] = 0.0
    x[11, :] = 0.0
    x[11, 5] = -3.0                                           # a row whose amax is one negative value
    codes, scales = oracle_mod.quantize_e4m3(x)
    assert scales[7] == 0 and not codes[7].any()
    amax = np.abs(x).max(axis=1)
    live = amax > 0
    assert np.array_equal(scales[live], (amax[live] / np.float32(448)).astype(np.float32))
    # each row's largest magnitude lands on the format's largest finite value
    arg = np.abs(x).argmax(axis=1)
    top = codes[np.arange(300), arg][live]
    assert np.all((top & 0x7F) == 0x7E)
    assert codes[11, 5] == 0xFE
    # every code is the nearest to x * (448 / amax): at most half a code step
    y = x[live] * (np.float32(448) / amax[live])[:, None]
    yv = oracle_mod.e4m3_to_double(codes[live])
    e = np.floor(np.log2(np.maximum(np.abs(y).astype(np.float64), 2.0 ** -6)))
    half_step = 2.0 ** (e - 3) / 2
    assert np.all(np.abs(y - yv) <= half_step * (1 + 1e-12))


def test_indexer_e4m3_worked_example(oracle_mod):
    g = golden("e4m3_worked.json")["scores"]
    q = bf16_bits(torch.tensor(g["q"], dtype=torch.float32)).reshape(1, 1, 4)
    w = np.array([g["w"]], np.float32)
    codes, sc = oracle_mod.quantize_e4m3(np.array(g["keys"], np.float32))
    got = oracle_mod.indexer_scores_e4m3(q, w, codes, sc, np.array([0, 4], np.int64))
    want = np.array([closed_form(e) for e in g["expected"]])
    assert np.allclose(got, want, rtol=g["rel_tol"], atol=0)
    assert got[1] == 0.0 and got[3] == 0.0


def test_indexer_e4m3_library_matmul_and_one_hot(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 2)
    B, Hi, Di = 3, 5, 64
    counts = [17, 0, 40]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    q_bits = _normal_bits("e4m3_q", (B, Hi, Di))
    w = rng.uniform(0, 1, (B, Hi)).astype(np.float32)
    kx = (rng.standard_normal((int(offs[-1]), Di)) * 3).astype(np.float32)
    kx[5] = 0.0
    kx[6] = 0.0
    kx[6, 9] = -2.5                                           # a one-hot key
    codes, sc = oracle_mod.quantize_e4m3(kx)
    got = oracle_mod.indexer_scores_e4m3(q_bits, w, codes, sc, offs)
    # numpy float64 on the dequantized operands (queries quantized per row)
    qc, qs = oracle_mod.quantize_e4m3(bf16_values(q_bits).reshape(-1, Di).astype(np.float32))
    qhat = oracle_mod.dequantize_e4m3(qc, qs).reshape(B, Hi, Di)
    khat = oracle_mod.dequantize_e4m3(codes, sc)
    for b in range(B):
        rows = slice(int(offs[b]), int(offs[b + 1]))
        want = np.maximum(khat[rows] @ qhat[b].T, 0.0) @ w[b].astype(np.float64)
        assert np.allclose(got[rows], want, rtol=1e-12, atol=1e-300)
    assert got[5] == 0.0
    # the one-hot key: sum_h w_h max(0, qhat[h, 9] * khat[6, 9])
    assert khat[6, 9] == pytest.approx(-2.5, rel=1e-6)
    want6 = sum(float(w[0, h]) * max(0.0, qhat[0, h, 9] * khat[6, 9]) for h in range(Hi))
    assert got[6] == pytest.approx(want6, rel=1e-12)


def test_layer_step_e4m3_key_pool_matches_bulk_compression_of_history(oracle_mod):
    """With an E4M3 key pool the step writes the completed block's indexer key
    as the per-row quantization of the fp32-rounded compressor output: after
    the step the pool equals the quantized bulk compression of the history,
    and the scores are the E4M3 scores over that pool."""
    shape = synth.TINY
    L = 64
    st, raw = synth.raw_token_state(RNG_SEED, 4, shape, L)
    s = _np_state(st)
    kvh = bf16_bits(raw["kv"])
    prefix = oracle_mod.compress(kvh, bf16_bits(raw["z"]), s["b_kv"], 4)[0]
    s["kv_pool"][:prefix.shape[0]] = oracle_mod.float_to_bf16(prefix.astype(np.float32))
    pk = oracle_mod.compress(bf16_bits(raw["ik"]), bf16_bits(raw["iz"]), s["b_ik"], 4)[0]
    cap = s["key_pool"].shape[0]
    s["key_fp8"] = True
    s["key_pool"] = np.zeros((cap, shape.Di), np.uint8)
    s["key_scale"] = np.zeros(cap, np.float32)
    c0, s0 = oracle_mod.quantize_e4m3(pk.astype(np.float32))
    s["key_pool"][:pk.shape[0]] = c0
    s["key_scale"][:pk.shape[0]] = s0
    res = oracle_mod.layer_decode(s)
    full_ik = np.concatenate([bf16_bits(raw["ik"])[0], s["ik_new"]], axis=0)[None]
    full_iz = np.concatenate([bf16_bits(raw["iz"])[0], s["iz_new"]], axis=0)[None]
    bulk = oracle_mod.compress(full_ik, full_iz, s["b_ik"], 4)[0].astype(np.float32)
    bc, bs = oracle_mod.quantize_e4m3(bulk)
    n = L // 4
    assert np.array_equal(s["key_pool"][:n], bc) and np.array_equal(s["key_scale"][:n], bs)
    want = oracle_mod.indexer_scores_e4m3(s["iq"], s["w"], bc, bs, np.array([0, n], np.int64))
    assert np.array_equal(res["scores64"], want)


# ---------------------------------------------------------------- multi-token queries

@pytest.mark.parametrize("kind,phase", [(4, 0), (4, 1), (4, 2), (4, 3),
                                        (128, 0), (128, 1), (128, 2), (128, 64)])
def test_layer_two_token_step_equals_two_single_token_steps(oracle_mod, kind, phase):
    """A step with T = 2 query tokens (the current token and a draft token of
    speculative decoding, verified together) gives each token exactly what
    decoding the two tokens one per step gives it: outputs, log-sum-exps,
    scores and selections, and the same pools and rings afterwards.  The
    phases put a block completion on the first token, on the second, or on
    neither."""
    shape = synth.TINY
    r = kind
    base = [4096, 384, 256] if kind == 4 else [8192, 1024, 256]
    L = torch.tensor([b + phase for b in base], dtype=torch.int32)   # tokens after the step
    st2 = synth.filled_state(RNG_SEED, kind, shape, L, name=f"mtp{kind}", T=2)
    s2 = _np_state(st2)
    s2["T"], s2["W"] = 2, shape.W
    s1 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in s2.items()}
    Lin = s2["seq_len_in"].astype(np.int64)
    s1["swa"] = oracle_mod._window_ring(s2["swa"], Lin, shape.W)
    s1["T"] = 1
    per_token = ["q", "kv_new", "z_new"] + (["ik_new", "iz_new", "iq", "w"] if kind == 4 else [])
    r2 = oracle_mod.layer_decode(s2)
    singles = []
    for t in range(2):
        for name in per_token:
            s1[name] = np.ascontiguousarray(s2[name][:, t])
        s1["seq_len_in"] = (Lin + t).astype(np.int32)
        singles.append(oracle_mod.layer_decode(s1))
    assert np.array_equal(r2["seq_len_out"], singles[1]["seq_len_out"])
    for t in range(2):
        a, b = r2["tokens"][t], singles[t]
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
        assert np.array_equal(r2["out"][:, t], b["out"])
        if kind == 4:
            assert np.array_equal(a["scores64"], b["scores64"])
            assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(r2["idx"][:, t], b["idx"])
    for name in ["kv_pool", "kv_ring", "z_ring"] + (["key_pool", "ik_ring", "iz_ring"] if kind == 4 else []):
        assert np.array_equal(s2[name], s1[name]), name
    Lout = Lin + 2
    assert np.array_equal(oracle_mod._window_ring(s2["swa"], Lout, shape.W),
                          oracle_mod._window_ring(s1["swa"], Lout, shape.W))
    # a block completed in the step: the pool's last live row was written in it
    done = [(int(Lin[b]) + t + 1) % r == 0 for b in range(3) for t in range(2)]
    assert any(done) == (phase in ((0, 1) if kind == 4 else (0, 1)))


# ---------------------------------------------------------------- C4 overlap transform

def test_compress_overlap_worked_example(oracle_mod):
    g = golden("compress_overlap_worked.json")
    kv = bf16_bits(np.array(g["kv"], np.float32)).reshape(1, -1, 1)
    z = bf16_bits(np.array(g["z"], np.float32)).reshape(1, -1, 1)
    b = np.array(g["b"], np.float32).reshape(-1, 1)
    got = oracle_mod.compress_overlap(kv, z, b, g["r"])[0, :, 0]
    want = np.array([closed_form(e) for e in g["expected"]])
    assert np.allclose(got, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("r", [1, 4, 7])
def test_compress_overlap_special_cases_reduce_to_the_compressor(oracle_mod, r):
    """A bias of -inf over the previous block's positions weighs it 0: the
    result is the (pinned) non-overlapping compressor with the bias of the
    block's own positions, bit for bit; entry 0 (no previous block) equals it
    for any bias."""
    S, T, C = 2, 9 * r + (r - 1), 24
    kv = _normal_bits(f"ov.kv{r}", (S, T, C))
    z = _normal_bits(f"ov.z{r}", (S, T, C))
    b = (np.random.default_rng(RNG_SEED + r).standard_normal((2 * r, C)) * 0.5).astype(np.float32)
    own = oracle_mod.compress(kv, z, np.ascontiguousarray(b[r:]), r)
    ov = oracle_mod.compress_overlap(kv, z, b, r)
    assert np.array_equal(ov[:, 0], own[:, 0])
    bm = b.copy()
    bm[:r] = -np.inf
    assert np.array_equal(oracle_mod.compress_overlap(kv, z, bm, r), own)


def test_compress_overlap_constant_gate_and_library_softmax(oracle_mod):
    r, S, T, C = 4, 2, 40, 16
    kv = _normal_bits("ov.kvc", (S, T, C))
    zeros = np.zeros((S, T, C), np.uint16)                   # bf16 +0.0
    got = oracle_mod.compress_overlap(kv, zeros, np.zeros((2 * r, C), np.float32), r)
    v = bf16_values(kv)
    for n in range(T // r):
        lo = max(0, n * r - r)
        assert np.allclose(got[:, n], v[:, lo:n * r + r].mean(axis=1), rtol=1e-13, atol=1e-15)
    z = _normal_bits("ov.zc", (S, T, C))
    b = (np.random.default_rng(RNG_SEED + 9).standard_normal((2 * r, C)) * 0.5).astype(np.float32)
    got = oracle_mod.compress_overlap(kv, z, b, r)
    zv = bf16_values(z)
    for n in range(T // r):
        lo = max(0, n * r - r)
        i0 = lo - (n * r - r)
        logits = zv[:, lo:n * r + r] + b[i0:].astype(np.float64)[None]
        wts = scipy.special.softmax(logits, axis=1)
        assert np.allclose(got[:, n], (wts * v[:, lo:n * r + r]).sum(axis=1), rtol=1e-12, atol=1e-14)
