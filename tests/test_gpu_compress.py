"""GPU parity of the Flash Compressor against the oracle (max relative error <= 5e-3)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu
SEED = synth.SEED["compress"]


def rel_err(gpu, ref):
    """Element-wise |g - r| / max(|r|, 1e-2) (floor for near-zero outputs)."""
    return np.abs(gpu - ref) / np.maximum(np.abs(ref), 1e-2)


def _inputs(S, T, C, r, tag):
    kv = synth.normal_bf16(SEED, f"t.kv.{tag}", (S, T, C))
    z = synth.normal_bf16(SEED, f"t.z.{tag}", (S, T, C))
    b = synth.normal(SEED, f"t.b.{tag}", (r, C), std=0.5)
    return kv, z, b


# besides the ratios and widths of the workloads: shared-memory stages that
# span two sequences (5 blocks a sequence, 4 a stage, 2 tail tokens each), one
# block a stage (r = 16, the longest staged block), the first lengths past it
# (r = 20, 33: one thread per chunk and block), the widest staged row (C = 768)
# and the first width past it (C = 776)
@pytest.mark.parametrize("S,T,C,r", [(2, 1024, 512, 4), (2, 1024, 512, 128), (3, 37, 24, 4),
                                     (1, 130, 64, 128), (2, 16, 8, 1), (1, 300, 16, 7),
                                     (4, 4096, 576, 4), (4, 4096, 128, 4), (3, 22, 512, 4),
                                     (2, 160, 256, 16), (2, 100, 64, 20), (2, 300, 576, 33),
                                     (2, 90, 768, 3), (1, 64, 776, 4)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_compress_matches_oracle(oracle_mod, S, T, C, r, out_dtype):
    kv, z, b = _inputs(S, T, C, r, f"{S}.{T}.{C}.{r}")
    out = _lib.hsa_compress(kv.cuda(), z.cuda(), b.cuda(), r, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle_mod.compress(bf16_bits(kv), bf16_bits(z), b.numpy(), r, threads=8)
    got = out.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    err = rel_err(got, ref)
    assert err.max() <= 5e-3, f"max rel err {err.max():.3e}"
    if out_dtype == torch.float32:
        assert err.max() <= 1e-4  # fp32 output: only fp32 arithmetic error remains


def test_compress_full_size_sampled(oracle_mod):
    """The standalone workload (32 x 65,536 x 512) at both ratios; the oracle
    checks a seeded sample of (sequence, block) outputs."""
    S, T, C = 32, 65536, 512
    kv = synth.normal_bf16(SEED, "compress.kv", (S, T, C), device="cuda")
    z = synth.normal_bf16(SEED, "compress.z", (S, T, C), device="cuda")
    for r in (4, 128):
        b = synth.normal(SEED, f"compress.b.{r}", (r, C), std=0.5, device="cuda")
        out = _lib.hsa_compress(kv, z, b, r)
        torch.cuda.synchronize()
        nblk = T // r
        picks = synth.randint(SEED, f"compress.sample.{r}", 24, 0, S * nblk - 1).tolist()
        picks += [0, S * nblk - 1]
        for p in picks:
            s, n = divmod(int(p), nblk)
            ref = oracle_mod.compress(bf16_bits(kv[s:s + 1, n * r:(n + 1) * r]),
                                      bf16_bits(z[s:s + 1, n * r:(n + 1) * r]),
                                      b.cpu().numpy(), r)[0, 0]
            got = out[s, n].float().cpu().numpy()
            assert rel_err(got, ref).max() <= 5e-3


def test_compress_empty_and_partial_blocks():
    kv = torch.zeros(2, 3, 16, dtype=torch.bfloat16, device="cuda")
    out = _lib.hsa_compress(kv, kv, torch.zeros(4, 16, device="cuda"), 4)
    assert out.shape == (2, 0, 16)


# ---------------------------------------------------------------- C4 overlap transform

@pytest.mark.parametrize("S,T,C,r", [(2, 1024, 512, 4), (3, 37, 24, 4), (1, 300, 16, 7),
                                     (2, 16, 8, 1), (1, 1024, 64, 128), (4, 4096, 576, 4)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_compress_overlap_matches_oracle(oracle_mod, S, T, C, r, out_dtype):
    """Entry n over the 2r-token window of blocks n-1 and n (entry 0 over
    block 0 alone), a bias per window position; ragged tails dropped."""
    kv, z, _ = _inputs(S, T, C, r, f"ov.{S}.{T}.{C}.{r}")
    b = synth.normal(SEED, f"t.bov.{S}.{T}.{C}.{r}", (2 * r, C), std=0.5)
    out = _lib.hsa_compress_overlap(kv.cuda(), z.cuda(), b.cuda(), r, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle_mod.compress_overlap(bf16_bits(kv), bf16_bits(z), b.numpy(), r, threads=8)
    got = out.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    err = rel_err(got, ref)
    assert err.max() <= 5e-3, f"max rel err {err.max():.3e}"
    if out_dtype == torch.float32:
        assert err.max() <= 1e-4


def test_compress_overlap_masked_previous_block(oracle_mod):
    """A bias of -inf over the previous block's window positions masks them:
    the result is the non-overlapping compressor's (GPU against the oracle of
    both forms)."""
    S, T, C, r = 2, 512, 64, 4
    kv, z, b = _inputs(S, T, C, r, "ovm")
    bm = torch.cat([torch.full((r, C), float("-inf")), b], 0).contiguous()
    out = _lib.hsa_compress_overlap(kv.cuda(), z.cuda(), bm.cuda(), r, out_dtype=torch.float32)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = oracle_mod.compress(bf16_bits(kv), bf16_bits(z), b.numpy(), r)
    assert np.array_equal(ref, oracle_mod.compress_overlap(bf16_bits(kv), bf16_bits(z), bm.numpy(), r))
    assert np.isfinite(got).all() and rel_err(got, ref).max() <= 1e-4


def test_compress_overlap_full_size_sampled(oracle_mod):
    """The standalone workload (32 x 65,536 x 512) with the overlap transform at
    r = 4; the oracle checks a seeded sample of (sequence, entry) outputs."""
    S, T, C, r = 32, 65536, 512, 4
    kv = synth.normal_bf16(SEED, "compress.kv", (S, T, C), device="cuda")
    z = synth.normal_bf16(SEED, "compress.z", (S, T, C), device="cuda")
    b = synth.normal(SEED, "compress.bov.4", (2 * r, C), std=0.5, device="cuda")
    out = _lib.hsa_compress_overlap(kv, z, b, r)
    torch.cuda.synchronize()
    nblk = T // r
    picks = synth.randint(SEED, "compress.sample.ov", 24, 0, S * nblk - 1).tolist() + [0, nblk, S * nblk - 1]
    for p in picks:
        s, n = divmod(int(p), nblk)
        lo = max(0, n - 1) * r
        ref = oracle_mod.compress_overlap(bf16_bits(kv[s:s + 1, lo:(n + 1) * r]),
                                          bf16_bits(z[s:s + 1, lo:(n + 1) * r]),
                                          b.cpu().numpy(), r)[0, -1]
        got = out[s, n].float().cpu().numpy()
        assert rel_err(got, ref).max() <= 5e-3
