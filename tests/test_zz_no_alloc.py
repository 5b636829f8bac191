"""The allocation-free top-k (hsa_topk_noalloc) against the workspace version.

hsa_topk_noalloc serves callers that own only their input and output buffers
and cannot hand the library a workspace (a framework-managed allocator, or a
path that must not call cudaMalloc).  Its scratch is a static device array
shared by every call, so this checks two calls in a row with different
shapes (the second must not see the first one's leftovers), each bit-exact
against hsa_topk with a caller workspace.  The file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from hybrid_sparse_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


def _rows(lens, tag):
    rows = [synth.topk_scores(synth.SEED["topk"], 1, n, 0.05)[0] for n in lens]
    rows.append(synth.pair_ties_at_top(rows[-1], 600))
    vals = torch.cat(rows).cuda()
    offs = torch.zeros(len(rows) + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(torch.tensor([r.numel() for r in rows]), 0)
    return vals, offs.cuda()


@pytest.mark.parametrize("k", [512, 64])
def test_noalloc_topk_matches_workspace_topk_twice(k):
    cases = [_rows([300000, 4096, 0, 7, 20000], "a"), _rows([1000, 65, 150000], "b")]
    for vals, offs in cases:                        # two calls in a row, different layouts
        ref_idx, ref_vals = _lib.hsa_topk(vals, offs, k)
        idx, v = _lib.hsa_topk_noalloc(vals, offs, k)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.equal(v, ref_vals)


def test_noalloc_topk_rejects_sizes_beyond_its_scratch():
    lib = _lib.load()
    fake = ctypes.c_void_p(0x1000)                  # never dereferenced: rejected first
    rc = lib.hsa_topk_noalloc(fake, fake, 64, 64 * 262144, 512, fake, None, None)
    assert rc == 2                                  # HSA_ERR_UNSUPPORTED
    assert b"static array holds" in lib.hsa_last_error_detail()
