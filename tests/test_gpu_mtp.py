"""Parity of the layer step with T = 2 query tokens per sequence (speculative
decoding with a one-layer multi-token-prediction head: the current token and a
draft token verified together) against the oracle's composition: per token its
indexer scores (within the accumulation bound), its top-k (bit-exact on the
GPU's own scores; set agreement with the oracle's own pipeline) and its
attention (the oracle fed the GPU's indices); the pools, rings and window
after the step."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, bf16_values, np_state, set_agreement
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu
T = 2


def _run(g, T=T):
    B, sh = g.seq_len_in.numel(), g.shape
    res = {"out": torch.empty(B, T, sh.Hq, sh.Dv, dtype=torch.bfloat16, device="cuda"),
           "lse": torch.empty(B, T, sh.Hq, dtype=torch.float32, device="cuda"),
           "seq_len_out": torch.empty_like(g.seq_len_in)}
    kw = {}
    if g.kind == 4:
        res["idx"] = torch.empty(B, T, sh.k, dtype=torch.int32, device="cuda")
        res["scores"] = torch.zeros(T, g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
        kw = dict(topk_idx=res["idx"], scores=res["scores"])
    desc = _lib.layer_desc(g, res["out"], res["lse"], res["seq_len_out"], **kw)
    assert desc.T == T
    ws = _lib.hsa_layer_decode(desc)
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    return res


def _score_tol(iq, w, keys, offs):
    q, k = np.abs(bf16_values(iq)), np.abs(bf16_values(keys))
    out = np.zeros(k.shape[0])
    for b in range(len(offs) - 1):
        lo, hi = int(offs[b]), int(offs[b + 1])
        out[lo:hi] = (k[lo:hi] @ q[b].T) @ np.abs(w[b].astype(np.float64))
    return 2.0 ** -7 * out + 1e-30


def _check(oracle_mod, g, s, res, ref, min_agree, T=T):
    kind = g.kind
    Lin = s["seq_len_in"].astype(np.int64)
    assert np.array_equal(res["seq_len_out"].cpu().numpy(), Lin + T)
    offs = s["pool_offsets"]
    # pools: every live row within the compressor tolerance (the oracle's own pools)
    cnt = (Lin + T) // kind
    gp, rp = bf16_values(bf16_bits(g.kv_pool.cpu())), bf16_values(s["kv_pool"])
    for b in range(len(Lin)):
        lo, n = int(offs[b]), int(cnt[b])
        if n:
            err = np.abs(gp[lo:lo + n] - rp[lo:lo + n]) / np.maximum(np.abs(rp[lo:lo + n]), 1e-2)
            assert err.max() <= 5e-3
    # the rings and the window: the appended rows are copies
    assert np.array_equal(bf16_bits(g.swa.cpu()), s["swa"])
    assert np.array_equal(bf16_bits(g.kv_ring.cpu()), s["kv_ring"])
    errs = []
    for t in range(T):
        Lt = Lin + t + 1
        counts = Lt // kind
        rt = ref["tokens"][t]
        idx_t = None
        if kind == 4:
            key_rows, key_offs = oracle_mod.compact(s["key_pool"], offs, counts)
            gs = res["scores"][t].cpu().numpy().astype(np.float64)
            got = np.concatenate([gs[int(offs[b]):int(offs[b]) + int(counts[b])]
                                  for b in range(len(Lin))])
            iq_t = np.ascontiguousarray(s["iq"][:, t])
            w_t = np.ascontiguousarray(s["w"][:, t])
            assert np.all(np.abs(got - rt["scores64"]) <= _score_tol(iq_t, w_t, key_rows, key_offs))
            idx_t = res["idx"][:, t].cpu().numpy()
            own, _ = oracle_mod.topk(got.astype(np.float32), key_offs, s["k"], threads=16)
            assert np.array_equal(idx_t, own)
            agree = set_agreement(idx_t, rt["idx"], counts, s["k"])
            assert agree >= min_agree, f"token {t}: top-k set agreement {agree:.5f}"
        kv_rows, kv_offs = oracle_mod.compact(s["kv_pool"], offs, counts)
        ring = oracle_mod._window_ring(s["swa"], Lt, s["W"])
        o_ref, l_ref = oracle_mod.decode_attn(np.ascontiguousarray(s["q"][:, t]), ring,
                                              Lt.astype(np.int32), s["W"], kv_rows, kv_offs,
                                              idx_t, s["scale"], s["Dv"], threads=16)
        go = res["out"][:, t].float().cpu().numpy()
        err = np.abs(go - o_ref).max()
        assert err <= 1e-2, f"token {t}: attention max abs err {err:.3e}"
        assert np.abs(res["lse"][:, t].cpu().numpy() - l_ref).max() <= 2.0 ** -8
        errs.append(err)
    return errs


@pytest.mark.parametrize("kind,phase", [(4, 0), (4, 1), (4, 2), (128, 0), (128, 1), (128, 5)])
def test_layer_two_tokens_tiny(oracle_mod, kind, phase):
    """Three sequences; the phases put a block completion on the first token,
    on the second, or on neither."""
    base = [4096, 384, 260] if kind == 4 else [8192, 1024, 256]
    L = torch.tensor([b + phase for b in base], dtype=torch.int32)
    g = synth.filled_state(synth.SEED["tiny"], kind, synth.TINY, L, device="cuda",
                           name=f"mtp{kind}", T=T)
    s = np_state(g)
    res = _run(g)
    ref = oracle_mod.layer_decode(s, threads=16)
    _check(oracle_mod, g, s, res, ref, min_agree=62 / 64)


@pytest.mark.parametrize("kind,tokens,phase", [(4, 3, 1), (4, 3, 3), (4, 4, 0), (4, 4, 3),
                                               (128, 3, 2), (128, 3, 0), (128, 4, 3),
                                               (128, 4, 1), (128, 4, 9)])
def test_layer_three_and_four_tokens_tiny(oracle_mod, kind, tokens, phase):
    """T = 3 and 4 (the most a step takes): a block completion on the first
    token (the later tokens then write the next block's first slots after the
    completed block is read), on the last, or on none."""
    base = [4096, 384, 260] if kind == 4 else [8192, 1024, 256]
    L = torch.tensor([b + phase for b in base], dtype=torch.int32)
    g = synth.filled_state(synth.SEED["tiny"], kind, synth.TINY, L, device="cuda",
                           name=f"mtp{kind}t{tokens}", T=tokens)
    s = np_state(g)
    res = _run(g, T=tokens)
    ref = oracle_mod.layer_decode(s, threads=16)
    _check(oracle_mod, g, s, res, ref, min_agree=62 / 64, T=tokens)


def test_layer_two_tokens_c4_full_128k_batch64(oracle_mod):
    """The bench workload with two query tokens per sequence: batch 64, contexts
    U[16384, 131072], 64 heads x 576, indexer 8 x 128 per token (16 query rows
    on the tensor cores), top-512, window 128."""
    L = synth.c4_lengths(synth.SEED["c4layer"], 64) + 1
    g = synth.filled_state(synth.SEED["c4layer"], 4, synth.FULL, L, device="cuda",
                           name="mtp_c4layer", T=T)
    s = np_state(g)
    res = _run(g)
    ref = oracle_mod.layer_decode(s, threads=16)
    _check(oracle_mod, g, s, res, ref, min_agree=0.999)
