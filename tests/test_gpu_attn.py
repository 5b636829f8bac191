"""GPU parity of the fused hybrid attention against the oracle fed the same
indices.

Tolerances (the pages give none; the library fixes them from its arithmetic):
  * output, unit-scale values (the workloads' N(0,1) rows): max abs error
    <= 1e-2 with fp32 output; with the default bf16 output the rounding of o
    adds at most u * |o| (u = 2^-8, bf16 unit roundoff), so the bound is
    1e-2 + u * (|o_ref| + 1e-2);
  * output, values scaled up: the kernel rounds each softmax weight p_t to
    bf16 (relative error <= u) before the value product and divides by the
    sum of the rounded weights, so its output is an exact weighted mean with
    weights perturbed by a factor (1 + d_t) / (1 + d_mean); the error in
    channel c is then at most u / (1 - u) * (max_t V_t[c] - min_t V_t[c]).
    Large-value cases allow 1e-2 plus that per-channel bound;
  * log-sum-exp: the sum of the rounded weights is within a factor (1 +- u)
    of the exact one, so |d lse| <= -log(1 - u) ~ 2^-8 (+1% for the ex2 /
    log2 approximations)."""
import math

import numpy as np
import pytest
import torch

from helpers import bf16_bits, closed_form, golden
from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu
SEED = synth.SEED["c4layer"]
OUT_TOL = 1e-2
U_BF16 = 2.0 ** -8
LSE_TOL = -math.log(1.0 - U_BF16) * 1.01


def _offsets(counts):
    offs = torch.zeros(len(counts) + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0)
    return offs


def _run(q, swa, L, extra, offs, idx, scale, Dv, max_rows=0, out_dtype=torch.bfloat16):
    out, lse = _lib.hsa_decode_attn(
        q.cuda(), swa.cuda(), L.cuda(), None if extra is None else extra.cuda(),
        None if offs is None else offs.cuda(), None if idx is None else idx.cuda(),
        max_extra_rows=max_rows, scale=scale, Dv=Dv, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, Dv):
    return oracle_mod.decode_attn(
        bf16_bits(q), bf16_bits(swa), L.numpy(), swa.shape[1],
        None if extra is None else bf16_bits(extra), None if offs is None else offs.numpy(),
        None if idx is None else idx.numpy(), scale, Dv, threads=16)


def _compare(got, want, tol=OUT_TOL):
    """Element-wise |o - o_ref| <= tol (a scalar or an array broadcast against o)."""
    o, l = got
    ro, rl = want
    tol = np.broadcast_to(np.asarray(tol, np.float64), o.shape)
    excess = np.abs(o - ro) - tol
    err = np.abs(o - ro).max() if o.size else 0.0
    if o.size and excess.max() > 0:
        at = np.unravel_index(np.argmax(excess), o.shape)
        raise AssertionError(f"abs err {abs(o[at] - ro[at]):.3e} > tol {tol[at]:.3e} at {at}: "
                             f"got {o[at]:.6f} want {ro[at]:.6f} (max abs err {err:.3e})")
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    if fin.any():
        lerr = np.abs(l[fin] - rl[fin]).max()
        assert lerr <= LSE_TOL, f"lse err {lerr:.3e}"
    return err


def _bf16_out_tol(ro, base=OUT_TOL):
    """Bound for bf16 outputs: the fp32 result's bound plus its rounding to bf16."""
    return base + U_BF16 * (np.abs(ro) + base)


def _value_spread_tol(swa, L, extra, offs, idx, Dv, base=OUT_TOL):
    """[B, 1, Dv] bound base + u / (1 - u) * (max_t V_t[c] - min_t V_t[c]) over each
    token's attended rows (window rows, then the listed or all compressed rows)."""
    B, W = swa.shape[0], swa.shape[1]
    tol = np.full((B, 1, Dv), base)
    for b in range(B):
        Lb = int(L[b])
        rows = [swa[b, p % W, :Dv].float() for p in range(max(0, Lb - W), Lb)]
        if extra is not None:
            o0, o1 = int(offs[b]), int(offs[b + 1])
            js = [int(j) for j in idx[b] if j >= 0] if idx is not None else range(o1 - o0)
            rows += [extra[o0 + j, :Dv].float() for j in js]
        if rows:
            V = torch.stack(rows)
            spread = (V.max(dim=0).values - V.min(dim=0).values).double().numpy()
            tol[b, 0] += U_BF16 / (1 - U_BF16) * spread
    return tol


def test_attention_worked_example_embedded(oracle_mod):
    """The hand-worked 3-channel example, zero-padded to 128 channels (padding
    adds nothing to any dot product) and checked against its closed form."""
    g = golden("attn_worked.json")
    D = 128

    def pad(rows):
        a = torch.zeros(len(rows), D)
        a[:, :3] = torch.tensor(rows)
        return a.to(torch.bfloat16)

    q = pad([g["q"]])[None]                     # [1, 1, 128]
    swa = pad(g["swa"])[None]
    extra = pad(g["extra"])
    offs = torch.tensor([0, 2], dtype=torch.int64)
    L = torch.tensor([g["seq_len"]], dtype=torch.int32)
    for idx, key in ((torch.tensor([g["idx"]], dtype=torch.int32), "expected_sparse"),
                     (None, "expected_dense")):
        o, l = _run(q, swa, L, extra, offs, idx, 1.0, 128, max_rows=2, out_dtype=torch.float32)
        want = [closed_form(e) for e in g[key]["out"]]
        np.testing.assert_allclose(o[0, 0, :2], want, atol=OUT_TOL)
        assert abs(l[0, 0] - closed_form(g[key]["lse"])) < LSE_TOL
        assert np.all(o[0, 0, 3:] == 0)  # channels past the example are zero padding


def _tiny_case(B=1, Hq=8, D=128, Dv=128, W=64, k=64, counts=(1024,), L=(4096,), tag="tiny"):
    offs = _offsets(list(counts))
    q = synth.normal_bf16(SEED, f"at.q.{tag}", (B, Hq, D))
    swa = synth.normal_bf16(SEED, f"at.swa.{tag}", (B, W, D))
    extra = synth.normal_bf16(SEED, f"at.ex.{tag}", (int(offs[-1]), D))
    idx = torch.full((B, k), -1, dtype=torch.int32)
    for b in range(B):
        n = counts[b]
        m = min(k, n)
        if m:
            perm = synth.permutation(SEED, f"at.idx.{tag}.{b}", n)[:m]
            idx[b, :m] = perm.to(torch.int32)
    return q, swa, torch.tensor(list(L), dtype=torch.int32), extra, offs, idx


def test_attention_tiny_config(oracle_mod):
    q, swa, L, extra, offs, idx = _tiny_case()
    scale = 1 / math.sqrt(128)
    for out_dtype in (torch.bfloat16, torch.float32):
        got = _run(q, swa, L, extra, offs, idx, scale, 128, out_dtype=out_dtype)
        _compare(got, _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 128))


def test_attention_full_heads_ragged_sparse(oracle_mod):
    """64 heads x 576 (512 latent + 64 rope), window 128, top-512 lists with -1
    padding and repeats; windows shorter than, equal to and longer than W."""
    counts = [2000, 100, 0, 5000, 513, 1]
    Ls = [8003, 40, 1, 130000, 128, 3]
    B = len(counts)
    q, swa, L, extra, offs, idx = _tiny_case(B, 64, 576, 512, 128, 512, counts, Ls, "full")
    idx[3, 100:110] = idx[3, 0]          # repeated entries count once each
    idx[0, 7] = -1                       # a hole in the middle of a list
    scale = 1 / math.sqrt(576)
    got = _run(q, swa, L, extra, offs, idx, scale, 512)
    _compare(got, _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 512))


def test_attention_dense_c128_with_splits(oracle_mod):
    """Dense mode over all compressed rows: long lists are split across CTAs and
    merged by the log-sum-exp combine."""
    counts = [4000, 37, 1000, 0]
    Ls = [4000 * 128 + 5, 37 * 128 + 127, 128000, 64]
    B = len(counts)
    q, swa, L, extra, offs, _ = _tiny_case(B, 64, 576, 512, 128, 1, counts, Ls, "dense")
    scale = 1 / math.sqrt(576)
    got = _run(q, swa, L, extra, offs, None, scale, 512, max_rows=max(counts))
    _compare(got, _oracle(oracle_mod, q, swa, L, extra, offs, None, scale, 512))


def test_attention_rescale_path(oracle_mod):
    """Later tiles carry much larger logits than the window tile, forcing the
    running maximum to move and O to be rescaled in TMEM; the first tile of one
    sequence is entirely masked.  Only the rope channels (512..575, keys but not
    values) are scaled up, so the values keep unit scale and the fixed 1e-2
    bound applies."""
    counts = [900, 900]
    q, swa, L, extra, offs, idx = _tiny_case(2, 64, 576, 512, 128, 512, counts, [5000, 5000], "resc")
    ramp = torch.ones(extra.shape[0], 576)
    ramp[:, 512:] = torch.linspace(0.5, 40.0, extra.shape[0])[:, None]
    extra = (extra.float() * ramp).to(torch.bfloat16)
    L[1] = 0                                     # no window: tile 0 = compressed rows only
    idx[1, :200] = -1                            # ... whose first 128 slots are all masked
    scale = 1 / math.sqrt(576)
    got = _run(q, swa, L, extra, offs, idx, scale, 512, out_dtype=torch.float32)
    _compare(got, _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 512))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attention_large_values_every_channel(oracle_mod, out_dtype):
    """Every channel of the pool rows (keys and values) grows along the pool,
    up to 6x, as in the rescale case before its values were narrowed to unit
    scale: the running maximum moves and O is rescaled, and the values reach
    ~25 in magnitude.  Checked against 1e-2 plus the bf16-weight bound
    u / (1 - u) * (max_t V_t[c] - min_t V_t[c]) per channel (plus the output's
    own rounding for bf16)."""
    counts = [900, 900]
    q, swa, L, extra, offs, idx = _tiny_case(2, 64, 576, 512, 128, 512, counts, [5000, 5000], "resc")
    extra = (extra.float() * torch.linspace(0.5, 6.0, extra.shape[0])[:, None]).to(torch.bfloat16)
    L[1] = 0
    idx[1, :200] = -1
    scale = 1 / math.sqrt(576)
    want = _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 512)
    tol = _value_spread_tol(swa, L, extra, offs, idx, 512)
    if out_dtype == torch.bfloat16:
        tol = tol + U_BF16 * (np.abs(want[0]) + tol)
    assert tol.max() > 0.1           # the bound really is wider than the unit-scale one
    got = _run(q, swa, L, extra, offs, idx, scale, 512, out_dtype=out_dtype)
    _compare(got, want, tol)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("splits", [2, 3, 4])
def test_attention_cluster_merge_dense(oracle_mod, splits):
    """Dense lists of at most 896 rows (8 tiles with the 128-row window): with
    B = SMs // splits, the splits of a token form one thread-block cluster and
    merge in shared memory (no partials in global memory: the workspace is the
    header alone); short sequences leave their later splits empty."""
    B = _sms() // splits
    base_c = [896, 0, 5, 300, 700, 129, 896, 64]
    base_l = [896 * 128 + 5, 3, 64, 300 * 128, 128000, 130, 896 * 128 + 127, 0]
    counts = [base_c[i % 8] for i in range(B)]
    Ls = [base_l[i % 8] for i in range(B)]
    assert _lib.hsa_decode_attn_workspace_size(B, 64, 576, 512, 128, 896) == 256
    q, swa, L, extra, offs, _ = _tiny_case(B, 64, 576, 512, 128, 1, counts, Ls, f"cl{splits}")
    scale = 1 / math.sqrt(576)
    want = _oracle(oracle_mod, q, swa, L, extra, offs, None, scale, 512)
    _compare(_run(q, swa, L, extra, offs, None, scale, 512, max_rows=896, out_dtype=torch.float32), want)


def test_attention_cluster_merge_sparse_rescale(oracle_mod):
    """Top-512 lists (5 tiles with the window) at B = SMs // 2: two splits per
    token merged in their cluster; ragged and padded lists, a hole, repeated
    entries, a token whose first tile is entirely masked, and rope logits that
    grow along the pool (the running maximum moves and O^T is rescaled)."""
    B = _sms() // 2
    base_c = [2000, 100, 0, 5000, 513, 1, 900, 900]
    base_l = [8003, 40, 1, 130000, 128, 3, 5000, 0]
    counts = [base_c[i % 8] for i in range(B)]
    Ls = [base_l[i % 8] for i in range(B)]
    assert _lib.hsa_decode_attn_workspace_size(B, 64, 576, 512, 128, 512) == 256
    q, swa, L, extra, offs, idx = _tiny_case(B, 64, 576, 512, 128, 512, counts, Ls, "clsp")
    ramp = torch.ones(extra.shape[0], 576)
    ramp[:, 512:] = torch.linspace(0.5, 40.0, extra.shape[0])[:, None]
    extra = (extra.float() * ramp).to(torch.bfloat16)
    idx[0, 7] = -1
    idx[3, 100:110] = idx[3, 0]
    idx[7, :200] = -1          # no window (L = 0): the first 128 slots are all masked
    scale = 1 / math.sqrt(576)
    got = _run(q, swa, L, extra, offs, idx, scale, 512, out_dtype=torch.float32)
    _compare(got, _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 512))


def test_attention_few_rows_bf16_output(oracle_mod):
    """Tokens that attend only a handful of rows (|o| up to ~4) with the
    default bf16 output, through both the single-CTA path and the two-split
    cluster merge: bound 1e-2 + u * (|o_ref| + 1e-2)."""
    base_c = [1, 0, 5, 3, 2, 0, 512, 4]
    base_l = [0, 1, 2, 3, 0, 7, 4, 1]
    for B in (8, _sms() // 2):
        counts = [base_c[i % 8] for i in range(B)]
        Ls = [base_l[i % 8] for i in range(B)]
        q, swa, L, extra, offs, idx = _tiny_case(B, 64, 576, 512, 128, 512, counts, Ls, f"few{B}")
        scale = 1 / math.sqrt(576)
        want = _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 512)
        got = _run(q, swa, L, extra, offs, idx, scale, 512)   # bf16 output (the default)
        assert np.abs(want[0]).max() > 1.5
        _compare(got, want, _bf16_out_tol(want[0]))


def test_attention_empty_and_window_only(oracle_mod):
    q, swa, L, extra, offs, idx = _tiny_case(3, 8, 128, 128, 64, 64, [10, 0, 5], [0, 0, 70], "empty")
    idx[0] = -1
    scale = 0.1
    got = _run(q, swa, L, extra, offs, idx, scale, 128)
    want = _oracle(oracle_mod, q, swa, L, extra, offs, idx, scale, 128)
    _compare(got, want)
    assert np.all(got[0][0] == 0) and np.all(np.isneginf(got[1][0]))
    # window only (no compressed pool at all)
    got = _run(q, swa, L, None, None, None, scale, 128)
    _compare(got, _oracle(oracle_mod, q, swa, L, None, None, None, scale, 128))


def test_attention_index_out_of_range_flags_bounds():
    q, swa, L, extra, offs, idx = _tiny_case(1, 8, 128, 128, 64, 64, [10], [100], "oob")
    idx[0, 3] = 10                                # sequence has 10 rows: 10 is out of range
    ws = _lib.workspace(_lib.hsa_decode_attn_workspace_size(1, 8, 128, 128, 64, 64))
    _lib.hsa_decode_attn(q.cuda(), swa.cuda(), L.cuda(), extra.cuda(), offs.cuda(), idx.cuda(),
                         Dv=128, ws=ws)
    assert _lib.hsa_workspace_status(ws) & 0x1
