"""Parity of the E4M3 indexer-key pool: the per-row quantizer (bit-exact), the
indexer over E4M3 keys (the oracle on the same codes), and the C4 layer step
with an E4M3 key pool (pools against the oracle's own quantization, scores,
top-k, attention).  The format: E4M3 codes with one fp32 scale per row
(scale = amax / 448), the score formula on the dequantized operands."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, bf16_values, np_state, set_agreement
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

SEED = 0xF8


def _gen(name, shape, std=1.0):
    return synth.normal(SEED, name, shape, std=std)


def e4m3_score_tol(oracle_mod, iq, w, codes, kscale, offs, factor=2.0 ** -17):
    """factor * sum_h w_h sum_d |qhat_hd khat_jd| per row: the fp32 accumulation
    bound of 128 exact E4M3 products (and the scale products after it)."""
    B, Hi, Di = iq.shape
    qc, qs = oracle_mod.quantize_e4m3(bf16_values(iq).reshape(-1, Di).astype(np.float32))
    qhat = np.abs(oracle_mod.dequantize_e4m3(qc, qs)).reshape(B, Hi, Di)
    khat = np.abs(oracle_mod.dequantize_e4m3(codes, kscale))
    out = np.zeros(codes.shape[0])
    for b in range(B):
        lo, hi = int(offs[b]), int(offs[b + 1])
        out[lo:hi] = (khat[lo:hi] @ qhat[b].T) @ np.abs(w[b].astype(np.float64))
    return factor * out + 1e-30


@pytest.mark.parametrize("C", [4, 128, 576])
def test_quantize_e4m3_bit_exact(oracle_mod, C):
    rows = 2000
    x = _gen(f"q{C}", (rows, C))
    scale = torch.exp(synth.normal(SEED, f"qs{C}", (rows, 1), std=4.0))   # amax from ~1e-5 to ~1e5
    x = (x * scale).contiguous()
    x[3] = 0.0                                         # a zero row
    x[5, :] = 2.0 ** -140                              # a subnormal-valued row
    x[7, 0] = -x[7].abs().max() * 2                    # amax on a negative entry
    codes, sc = _lib.hsa_quantize_e4m3(x.cuda())
    torch.cuda.synchronize()
    want_c, want_s = oracle_mod.quantize_e4m3(x.numpy())
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), want_s.view(np.uint32))


def test_quantize_e4m3_ties_round_to_even(oracle_mod):
    """Rows whose scaled entries land exactly on midpoints between codes
    (amax = 448, so x * 448 / amax = x): every tie goes to the even code."""
    vals = oracle_mod.e4m3_to_double(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    n = len(mids)
    C = 128
    rows = (n + C - 2) // (C - 1)
    x = np.zeros((rows, C), np.float32)
    x[:, 0] = 448.0
    flat = np.concatenate([mids, np.zeros(rows * (C - 1) - n, np.float32)])
    x[:, 1:] = flat.reshape(rows, C - 1) * np.where(np.arange(rows) % 2 == 0, 1, -1)[:, None]
    codes, sc = _lib.hsa_quantize_e4m3(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    want_c, want_s = oracle_mod.quantize_e4m3(x)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(sc.cpu().numpy(), want_s)


def _pool(oracle_mod, name, counts, Di=128, std=1.0):
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    x = _gen(name, (int(offs[-1]), Di), std=std)
    codes, sc = oracle_mod.quantize_e4m3(x.numpy())
    gcodes, gsc = _lib.hsa_quantize_e4m3(x.cuda())
    return offs, codes, sc, gcodes, gsc


@pytest.mark.parametrize("Hi", [1, 3, 8, 16])
def test_indexer_e4m3_ragged(oracle_mod, Hi):
    """Ragged sequences (empty, shorter than a tile, several tiles and a ragged
    tail), many short sequences per CTA (the query buffers cycle)."""
    counts = [0, 1, 127, 128, 129, 1000, 0, 5000, 3] + [17] * 600 + [300]
    B = len(counts)
    offs, codes, sc, gcodes, gsc = _pool(oracle_mod, f"k{Hi}", counts)
    assert np.array_equal(gcodes.cpu().numpy(), codes)
    iq = synth.normal_bf16(SEED, f"iq{Hi}", (B, Hi, 128))
    w = synth.uniform(SEED, f"w{Hi}", (B, Hi))
    got = _lib.hsa_indexer_scores_e4m3(iq.cuda(), w.cuda(), gcodes, gsc,
                                       torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    want = oracle_mod.indexer_scores_e4m3(bf16_bits(iq), w.numpy(), codes, sc, offs, threads=16)
    tol = e4m3_score_tol(oracle_mod, bf16_bits(iq), w.numpy(), codes, sc, offs)
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= tol), f"max err / tol {np.max(err / tol):.3f}"


def test_indexer_e4m3_queries_with_large_and_zero_rows(oracle_mod):
    """Query rows of very different magnitudes, an all-zero query row (scale 0:
    that head adds nothing) and negative weights."""
    counts = [300, 700]
    B, Hi = 2, 8
    offs, codes, sc, gcodes, gsc = _pool(oracle_mod, "kz", counts, std=3.0)
    q = synth.normal(SEED, "iqz", (B, Hi, 128)) * torch.tensor([1e-3, 1, 50, 1e3] * 2)[None, :, None]
    q[1, 2] = 0.0
    iq = q.to(torch.bfloat16)
    w = synth.uniform(SEED, "wz", (B, Hi)) - 0.3
    got = _lib.hsa_indexer_scores_e4m3(iq.cuda(), w.cuda(), gcodes, gsc,
                                       torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    want = oracle_mod.indexer_scores_e4m3(bf16_bits(iq), w.numpy(), codes, sc, offs)
    tol = e4m3_score_tol(oracle_mod, bf16_bits(iq), w.numpy(), codes, sc, offs)
    assert np.all(np.abs(got.cpu().numpy() - want) <= tol)


def _to_e4m3_keys(oracle_mod, g, s):
    """The state's key pool as E4M3: the GPU quantizes its copy with the
    library, the oracle its own copy with its own quantizer (same fp32 input:
    the pool's bf16 values)."""
    kp = g.key_pool.float()
    g.key_pool, g.key_scale = _lib.hsa_quantize_e4m3(kp)
    codes, sc = oracle_mod.quantize_e4m3(bf16_values(s["key_pool"]).astype(np.float32), threads=16)
    s["key_pool"], s["key_scale"], s["key_fp8"] = codes, sc, True
    torch.cuda.synchronize()
    assert np.array_equal(g.key_pool.cpu().numpy(), codes)
    assert np.array_equal(g.key_scale.cpu().numpy(), sc)


def _run_step(g):
    B, sh = g.seq_len_in.numel(), g.shape
    res = {"out": torch.empty(B, sh.Hq, sh.Dv, dtype=torch.bfloat16, device="cuda"),
           "lse": torch.empty(B, sh.Hq, dtype=torch.float32, device="cuda"),
           "seq_len_out": torch.empty_like(g.seq_len_in),
           "idx": torch.empty(B, sh.k, dtype=torch.int32, device="cuda"),
           "scores": torch.zeros(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")}
    desc = _lib.layer_desc(g, res["out"], res["lse"], res["seq_len_out"], topk_idx=res["idx"],
                           scores=res["scores"])
    ws = _lib.hsa_layer_decode(desc)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    return res


def _check_step(oracle_mod, g, s, res, ref, min_agree, max_code_flips):
    L = ref["seq_len_out"].astype(np.int64)
    offs = s["pool_offsets"]
    counts = L // 4
    # the appended E4M3 key rows: the GPU quantized its fp32 compressor output,
    # the oracle its fp64 output rounded to fp32; the two fp32 values may
    # differ in the last bits, which can move a code by one step
    gk = g.key_pool.cpu().numpy()
    gsc = g.key_scale.cpu().numpy()
    new_rows = [int(offs[b]) + int(counts[b]) - 1 for b in range(len(L)) if L[b] % 4 == 0]
    if new_rows:
        dv = np.abs(oracle_mod.dequantize_e4m3(gk[new_rows], gsc[new_rows]) -
                    oracle_mod.dequantize_e4m3(s["key_pool"][new_rows], s["key_scale"][new_rows]))
        flips = int(np.sum(gk[new_rows] != s["key_pool"][new_rows]))
        assert flips <= max_code_flips, f"{flips} appended codes differ"
        # within one code step: 2^-3 of the entry's magnitude, or a subnormal step
        step = np.maximum(np.abs(oracle_mod.dequantize_e4m3(s["key_pool"][new_rows],
                                                            s["key_scale"][new_rows])) * 2.0 ** -3,
                          s["key_scale"][new_rows][:, None].astype(np.float64) * 2.0 ** -9)
        assert np.all(dv <= step * 1.0001 + 1e-30)
    # scores: the oracle's E4M3 scores over the GPU's own pool (identical codes)
    key_rows, key_offs = oracle_mod.compact(gk, offs, counts)
    ksc, _ = oracle_mod.compact(gsc.reshape(-1, 1), offs, counts)
    ksc = ksc.reshape(-1)
    want = oracle_mod.indexer_scores_e4m3(s["iq"], s["w"], key_rows, ksc, key_offs, threads=16)
    gs = res["scores"].cpu().numpy().astype(np.float64)
    got = np.concatenate([gs[int(offs[b]):int(offs[b]) + int(counts[b])] for b in range(len(L))])
    tol = e4m3_score_tol(oracle_mod, s["iq"], s["w"], key_rows, ksc, key_offs)
    assert np.all(np.abs(got - want) <= tol)
    # top-k bit-exact on the GPU's own scores; set agreement with the oracle's
    # own pipeline (its own pools and scores)
    gidx = res["idx"].cpu().numpy()
    own, _ = oracle_mod.topk(got.astype(np.float32), key_offs, s["k"], threads=16)
    assert np.array_equal(gidx, own)
    agree = set_agreement(gidx, ref["idx"], counts, s["k"])
    assert agree >= min_agree, f"top-k set agreement {agree:.5f}"
    # attention: the oracle fed the GPU's selected indices
    kv_rows, kv_offs = oracle_mod.compact(s["kv_pool"], offs, counts)
    o_ref, l_ref = oracle_mod.decode_attn(s["q"], s["swa"], L.astype(np.int32), s["swa"].shape[1],
                                          kv_rows, kv_offs, gidx, s["scale"], s["Dv"], threads=16)
    err = np.abs(res["out"].float().cpu().numpy() - o_ref).max()
    assert err <= 1e-2, f"attention max abs err {err:.3e}"
    assert np.abs(res["lse"].cpu().numpy() - l_ref).max() <= 2.0 ** -8


def test_layer_e4m3_keys_from_raw_tokens(oracle_mod):
    """One sequence from raw tokens (Hi = 2, Di = 128): each side compresses the
    history to fp32 and quantizes its own key pool; the step completes a block."""
    shape = synth.LayerShape(Hq=8, Dqk=128, Dv=128, Hi=2, Di=128, k=64, W=64)
    st, raw = synth.raw_token_state(SEED, 4, shape, 4096)
    s = np_state(st)
    pre = oracle_mod.compress(bf16_bits(raw["kv"]), bf16_bits(raw["z"]), s["b_kv"], 4)[0]
    s["kv_pool"][:pre.shape[0]] = oracle_mod.float_to_bf16(pre.astype(np.float32))
    pk = oracle_mod.compress(bf16_bits(raw["ik"]), bf16_bits(raw["iz"]), s["b_ik"], 4)[0]
    cap = s["key_pool"].shape[0]
    codes, sc = oracle_mod.quantize_e4m3(pk.astype(np.float32))
    s["key_pool"] = np.zeros((cap, 128), np.uint8)
    s["key_scale"] = np.zeros(cap, np.float32)
    s["key_pool"][:pk.shape[0]], s["key_scale"][:pk.shape[0]] = codes, sc
    s["key_fp8"] = True
    g = st.to("cuda")
    kv = _lib.hsa_compress(raw["kv"].cuda(), raw["z"].cuda(), g.b_kv, 4)
    g.kv_pool[:kv.shape[1]] = kv[0]
    ks = _lib.hsa_compress(raw["ik"].cuda(), raw["iz"].cuda(), g.b_ik, 4, out_dtype=torch.float32)
    g.key_pool = torch.zeros(cap, 128, dtype=torch.uint8, device="cuda")
    g.key_scale = torch.zeros(cap, dtype=torch.float32, device="cuda")
    gc, gsc = _lib.hsa_quantize_e4m3(ks[0].contiguous())
    g.key_pool[:gc.shape[0]] = gc
    g.key_scale[:gc.shape[0]] = gsc
    torch.cuda.synchronize()
    flips = int(np.sum(g.key_pool[:pk.shape[0]].cpu().numpy() != codes))
    assert flips <= pk.size // 1000, f"{flips} prefix codes differ"
    ref = oracle_mod.layer_decode(s)
    res = _run_step(g)
    _check_step(oracle_mod, g, s, res, ref, min_agree=62 / 64, max_code_flips=2)


def test_layer_e4m3_keys_c4_full_128k_batch64(oracle_mod):
    """The headline workload with an E4M3 key pool: batch 64, contexts
    U[16384, 131072], 64 heads x 576, indexer 8 x 128, top-512, window 128."""
    L = synth.c4_lengths(synth.SEED["c4layer"], 64)
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda")
    s = np_state(g)
    _to_e4m3_keys(oracle_mod, g, s)
    res = _run_step(g)
    ref = oracle_mod.layer_decode(s, threads=16)
    _check_step(oracle_mod, g, s, res, ref, min_agree=0.999, max_code_flips=64)
