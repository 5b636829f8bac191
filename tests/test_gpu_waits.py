"""The bounded waits of the indexer kernel: with the pipeline waits' bound
lowered to one check, a wait whose phase is not complete at once runs out; the
call then sets HSA_DEV_TIMEOUT, the kernel stops cleanly (the loads and MMAs it
issued are waited for, its TMEM freed) and returns, and the next call with the
default bound on the same stream is correct.  Nothing faults or hangs: the
abort is the kernel's own bounded path."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, bf16_values
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu
SEED = 0x5A17
HSA_DEV_TIMEOUT = 0x2


def _tol(iq, w, kv, offs):
    """1e-4 * sum_h |w_h| sum_d |q_hd k_jd| (k as float64 values)."""
    q = np.abs(bf16_values(bf16_bits(iq)))
    out = np.zeros(kv.shape[0])
    for b in range(len(offs) - 1):
        lo, hi = int(offs[b]), int(offs[b + 1])
        out[lo:hi] = (np.abs(kv[lo:hi]) @ q[b].T) @ np.abs(w[b].numpy().astype(np.float64))
    return 1e-4 * out + 1e-30


@pytest.mark.parametrize("fp8", [False, True])
def test_indexer_wait_runs_out_then_next_call_is_correct(oracle_mod, fp8):
    # ~272K entries: every CTA has more tiles than stages, so its producer
    # waits for a stage to be freed right after issuing its first loads (a
    # phase that cannot be complete that soon)
    counts = [100000, 0, 100000, 72000, 512]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    B, Hi, Di = len(counts), 8, 128
    iq = synth.normal_bf16(SEED, "w.q", (B, Hi, Di))
    w = synth.uniform(SEED, "w.w", (B, Hi))
    kx = synth.normal(SEED, "w.k", (int(offs[-1]), Di))
    d_offs = torch.from_numpy(offs).cuda()
    ws = _lib.workspace(_lib.hsa_indexer_scores_workspace_size())
    scores = torch.zeros(int(offs[-1]), dtype=torch.float32, device="cuda")
    if fp8:
        codes, sc = oracle_mod.quantize_e4m3(kx.numpy())
        gk, gs = _lib.hsa_quantize_e4m3(kx.cuda())
        run = lambda: _lib.hsa_indexer_scores_e4m3(iq.cuda(), w.cuda(), gk, gs, d_offs, scores, ws)
        want = oracle_mod.indexer_scores_e4m3(bf16_bits(iq), w.numpy(), codes, sc, offs)
        kv = oracle_mod.dequantize_e4m3(codes, sc)
    else:
        keys = kx.to(torch.bfloat16)
        run = lambda: _lib.hsa_indexer_scores(iq.cuda(), w.cuda(), keys.cuda(), d_offs, scores, ws)
        want = oracle_mod.indexer_scores(bf16_bits(iq), w.numpy(), bf16_bits(keys), offs)
        kv = bf16_values(bf16_bits(keys))
    torch.cuda.synchronize()
    _lib.hsa_set_wait_limit(nanos=10_000_000, polls=1)
    try:
        for _ in range(3):
            run()
            torch.cuda.synchronize()
            assert _lib.hsa_workspace_status(ws) & HSA_DEV_TIMEOUT
    finally:
        _lib.hsa_set_wait_limit(0, 0)
    scores.zero_()
    run()
    torch.cuda.synchronize()
    assert _lib.hsa_workspace_status(ws) == 0
    err = np.abs(scores.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= _tol(iq, w, kv, offs))
