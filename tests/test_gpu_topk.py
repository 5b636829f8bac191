"""GPU parity of Lightning TopK: indices bit-exact against the oracle on the same
fp32 scores (value descending, lower index first among equal values)."""
import numpy as np
import pytest
import torch

from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu
SEED = synth.SEED["topk"]


def _ragged(rows):
    vals = torch.cat([torch.as_tensor(r, dtype=torch.float32).reshape(-1) for r in rows]) \
        if rows else torch.zeros(0)
    offs = torch.zeros(len(rows) + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(torch.tensor([len(r) for r in rows], dtype=torch.int64), 0)
    return vals, offs


def _check(oracle_mod, vals, offs, k, ws=None):
    idx, v = _lib.hsa_topk(vals.cuda(), offs.cuda(), k, ws=ws)
    torch.cuda.synchronize()
    ref_idx, ref_v = oracle_mod.topk(vals.numpy(), offs.numpy(), k, threads=8)
    got = idx.cpu().numpy()
    bad = np.nonzero((got != ref_idx).any(axis=1))[0]
    assert bad.size == 0, f"rows {bad[:5]} differ: got {got[bad[0]][:12]} want {ref_idx[bad[0]][:12]}"
    gv, rv = v.cpu().numpy(), ref_v
    assert np.array_equal(gv, rv) or np.array_equal(np.isneginf(gv), np.isneginf(rv))
    return got


def test_topk_worked_example(oracle_mod):
    from helpers import golden
    g = golden("topk_worked.json")
    vals, offs = _ragged([[float(x) for x in r] for r in g["rows"]])
    for case in g["cases"]:
        idx, _ = _lib.hsa_topk(vals.cuda(), offs.cuda(), case["k"])
        assert idx.cpu().tolist() == case["expected"]


@pytest.mark.parametrize("k", [1, 64, 512, 2048])
def test_topk_ragged_rows_with_ties(oracle_mod, k):
    # ragged lengths across one and many 4,096-score compaction blocks and chunks
    lens = [0, 1, 5, 63, 64, 65, 511, 512, 513, 2047, 4096, 5000, 20000, 32768, 32769, 40000]
    rows = [synth.topk_scores(SEED, 1, n, 0.05)[0] for n in lens]
    rows.append(synth.pair_ties_at_top(rows[-1], 600))   # ties at the threshold, long row
    rows.append(synth.pair_ties_at_top(rows[12], 600))   # ... and in a short row
    rows.append(torch.round(rows[12] * 8) / 8)            # heavy duplicates, short row
    rows.append(torch.round(rows[-4] * 8) / 8)            # heavy duplicates, long row
    vals, offs = _ragged(rows)
    _check(oracle_mod, vals, offs, k)


def test_topk_special_values(oracle_mod):
    n = 3000
    equal = torch.full((n,), 0.25)
    rev = torch.arange(n, dtype=torch.float32).flip(0)
    zeros = torch.where(torch.arange(n) % 3 == 0, torch.tensor(-0.0), torch.tensor(0.0))
    infs = torch.full((n,), float("-inf"))
    infs[[7, 1500, 2999]] = float("inf")
    mixed = synth.normal(SEED, "topk.mixed", (n,))
    mixed[::5] = float("inf")
    mixed[1::7] = float("-inf")
    mixed[2::11] = -0.0
    tiny = torch.tensor([1e-45, -1e-45, 0.0, -0.0, 1.17549435e-38, -1.17549435e-38] * 100)
    # rows whose boundary bin after two digits holds more candidates than the
    # final CTA stages in shared memory (selection over the global candidates)
    equal_big = torch.full((20000,), 1.5)
    zeros_big = torch.where(torch.arange(32768) % 2 == 0, torch.tensor(-0.0), torch.tensor(0.0))
    vals, offs = _ragged([equal, rev, zeros, infs, mixed, tiny, equal_big, zeros_big])
    for k in (1, 100, 512):
        _check(oracle_mod, vals, offs, k)


@pytest.mark.parametrize("k", [1, 64, 512, 2048])
def test_topk_single_launch_rows(oracle_mod, k):
    """At most 32,768 scores in all: one clustered launch (a row spans up to
    four CTAs of 8,192 scores); ragged rows across the CTA slices, ties."""
    lens = [0, 1, 5, 511, 512, 513, 2047, 4095, 8191, 8193]
    rows = [synth.topk_scores(SEED, 1, n, 0.05)[0] for n in lens]
    rows.append(synth.pair_ties_at_top(rows[6], 600))
    rows.append(torch.round(rows[6] * 8) / 8)
    vals, offs = _ragged(rows)
    assert vals.numel() <= 32768
    _check(oracle_mod, vals, offs, k)


def test_topk_single_launch_full_row_and_heavy_ties(oracle_mod):
    """One row of exactly 32,768 (all four CTA slices full); then rows whose
    threshold bin outgrows the shared lists (candidates through the workspace)."""
    x = synth.pair_ties_at_top(synth.topk_scores(SEED, 1, 32768, 0.05)[0], 600)
    vals, offs = _ragged([x])
    for k in (512, 2048):
        _check(oracle_mod, vals, offs, k)
    equal = torch.full((20000,), 1.5)
    zeros = torch.where(torch.arange(12000) % 2 == 0, torch.tensor(-0.0), torch.tensor(0.0))
    vals, offs = _ragged([equal, zeros])
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(2, vals.numel(), 512))
    for k in (1, 100, 512):
        for _ in range(2):     # the workspace is left reusable
            _check(oracle_mod, vals, offs, k, ws=ws)


@pytest.mark.parametrize("k", [1, 512, 2048])
def test_topk_rising_rows(oracle_mod, k):
    """Long rows whose scores keep rising, so each new stage of a chunk passes
    the bar its earlier stages set (every score is counted and kept, then
    pruned); a sawtooth and a rising run with plateaus of equal values."""
    up = torch.arange(90000, dtype=torch.float32) * 1e-3
    saw = (torch.arange(70000) % 5000).to(torch.float32)
    steps = torch.floor(torch.arange(80000, dtype=torch.float32) / 300)
    vals, offs = _ragged([up, saw, steps, up.flip(0)])
    _check(oracle_mod, vals, offs, k)


def test_topk_same_workspace_reused(oracle_mod):
    rows = [synth.topk_scores(SEED, 1, n, 0.05)[0] for n in (10000, 3, 70000)]
    vals, offs = _ragged(rows)
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(3, vals.numel(), 512))
    for _ in range(3):
        _check(oracle_mod, vals, offs, 512, ws=ws)
    assert _lib.hsa_workspace_status(ws) == 0


def test_topk_full_size_64_rows_of_262144(oracle_mod):
    """The standalone workload: 64 x 262,144 fp32 with 5% copied entries, k=512,
    plus the adversarial row with ties at the threshold; every row bit-exact."""
    x = synth.topk_scores(SEED, 64, 262144, 0.05)
    x[5] = synth.pair_ties_at_top(x[5], 600)
    offs = torch.arange(65, dtype=torch.int64) * 262144
    _check(oracle_mod, x.reshape(-1), offs, 512)


@pytest.mark.parametrize("k", [512, 2048])
def test_topk_few_long_rows_many_pieces(oracle_mod, k):
    """4 rows x 262,144 (the C4 length of a 1M-token context): each row is cut
    into many pieces, whose CTAs also prune at the row's counts so far; one row
    with ties at the threshold and one with heavy duplicates."""
    x = synth.topk_scores(SEED, 4, 262144, 0.05)
    x[1] = synth.pair_ties_at_top(x[1], 600)
    x[2] = torch.round(x[2] * 16) / 16
    offs = torch.arange(5, dtype=torch.int64) * 262144
    _check(oracle_mod, x.reshape(-1), offs, k)


def test_topk_nan_sets_status_without_fault():
    vals = torch.tensor([1.0, float("nan"), 2.0, 3.0, 4.0] * 100)
    offs = torch.tensor([0, 500], dtype=torch.int64)
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(1, 500, 4))
    _lib.hsa_topk(vals.cuda(), offs.cuda(), 4, ws=ws)
    assert _lib.hsa_workspace_status(ws) & 0x4


def test_topk_bad_offsets_flag_bounds():
    vals = torch.randn(100).cuda()
    offs = torch.tensor([0, 50, 200], dtype=torch.int64).cuda()   # past the 100 scores
    ws = _lib.workspace(_lib.hsa_topk_workspace_size(2, 100, 8))
    idx, _ = _lib.hsa_topk(vals, offs, 8, ws=ws)
    assert _lib.hsa_workspace_status(ws) & 0x1
    assert (idx[1] == -1).all()
