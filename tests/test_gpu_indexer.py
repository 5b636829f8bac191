"""GPU parity of the tcgen05 indexer scores against the oracle.

Tolerance (derived from the arithmetic): bf16 products are exact in fp32 and
the fp32 accumulation of Di terms errs by at most ~Di * 2^-24 of the sum of
the absolute products, so every score must satisfy
    |s_gpu - s_ref| <= 1e-4 * sum_h |w_h| * sum_d |q_hd k_jd| + 1e-30."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, bf16_values
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu
SEED = synth.SEED["c4layer"]


def _offsets(counts):
    offs = torch.zeros(len(counts) + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0)
    return offs


def _bound(iq, w, keys, offs):
    q, k = np.abs(bf16_values(bf16_bits(iq))), np.abs(bf16_values(bf16_bits(keys)))
    wa = np.abs(w.numpy().astype(np.float64))
    out = np.zeros(k.shape[0])
    for b in range(len(offs) - 1):
        lo, hi = int(offs[b]), int(offs[b + 1])
        out[lo:hi] = (k[lo:hi] @ q[b].T) @ wa[b]
    return out


def _check(oracle_mod, iq, w, keys, offs):
    s = _lib.hsa_indexer_scores(iq.cuda(), w.cuda(), keys.cuda(), offs.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.indexer_scores(bf16_bits(iq), w.numpy(), bf16_bits(keys), offs.numpy(),
                                    threads=16)
    got = s.cpu().numpy().astype(np.float64)
    tol = 1e-4 * _bound(iq, w, keys, offs) + 1e-30
    err = np.abs(got - ref)
    worst = int(np.argmax(err - tol))
    assert np.all(err <= tol), f"row {worst}: got {got[worst]} want {ref[worst]} tol {tol[worst]}"
    return got, ref


@pytest.mark.parametrize("Hi,Di", [(2, 32), (8, 128), (8, 64), (16, 128), (1, 32)])
def test_indexer_ragged_matches_oracle(oracle_mod, Hi, Di):
    counts = [0, 1, 127, 128, 129, 300, 1024, 5, 2000]
    offs = _offsets(counts)
    B = len(counts)
    iq = synth.normal_bf16(SEED, f"ix.q.{Hi}.{Di}", (B, Hi, Di))
    w = synth.uniform(SEED, f"ix.w.{Hi}.{Di}", (B, Hi))
    keys = synth.normal_bf16(SEED, f"ix.k.{Hi}.{Di}", (int(offs[-1]), Di))
    _check(oracle_mod, iq, w, keys, offs)


def test_indexer_one_hot_exact(oracle_mod):
    """w one-hot and q one-hot: each score is w * relu(one key element), exactly."""
    B, Hi, Di, n = 3, 8, 128, 700
    offs = _offsets([n] * B)
    keys = synth.normal_bf16(SEED, "ix.oh.k", (B * n, Di))
    iq = torch.zeros(B, Hi, Di, dtype=torch.bfloat16)
    w = torch.zeros(B, Hi)
    for b in range(B):
        iq[b, b + 2, 17 * b + 3] = 1.0
        w[b, b + 2] = 0.5
    s = _lib.hsa_indexer_scores(iq.cuda(), w.cuda(), keys.cuda(), offs.cuda()).cpu()
    for b in range(B):
        col = keys[b * n:(b + 1) * n, 17 * b + 3].float()
        assert torch.equal(s[b * n:(b + 1) * n], 0.5 * torch.clamp(col, min=0))


def test_indexer_full_c4_layer_workload(oracle_mod):
    """The 128K-context batch-64 layer: 8 heads x 128 dims over every C4 entry
    (context lengths U[16384, 131072], entries = L/4), all rows checked."""
    L = synth.c4_lengths(SEED, 64)
    counts = (L.to(torch.int64) // 4).tolist()
    offs = _offsets(counts)
    total = int(offs[-1])
    keys = synth.normal_bf16(SEED, "c4layer.key_pool.dense", (total, 128), device="cuda")
    iq = synth.normal_bf16(SEED, "c4layer.iq", (64, 8, 128), device="cuda")
    w = synth.uniform(SEED, "c4layer.w", (64, 8), device="cuda")
    _check(oracle_mod, iq.cpu(), w.cpu(), keys.cpu(), offs)


def test_indexer_leaves_rows_outside_sequences_untouched():
    offs = torch.tensor([5, 100, 100, 260], dtype=torch.int64)   # rows 0-4 belong to nobody
    keys = synth.normal_bf16(SEED, "ix.gap.k", (300, 32)).cuda()
    iq = synth.normal_bf16(SEED, "ix.gap.q", (3, 2, 32)).cuda()
    w = torch.ones(3, 2).cuda()
    scores = torch.full((300,), -7.0, device="cuda")
    _lib.hsa_indexer_scores(iq, w, keys, offs.cuda(), scores=scores)
    s = scores.cpu()
    assert torch.all(s[:5] == -7.0) and torch.all(s[260:] == -7.0)
    assert torch.all(s[5:260] >= 0)
