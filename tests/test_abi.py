"""The C-ABI library loads and exports every entry point include/hsa.h declares;
host-side validation rejects bad arguments before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from hybrid_sparse_attention_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "hsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hsa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("hsa_compress", "hsa_topk", "hsa_topk_workspace_size", "hsa_status_string",
                     "hsa_workspace_status", "hsa_last_error_detail"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []
    # the binding describes every declared function
    assert sorted(_lib.SIGNATURES) == declared_functions()


def test_status_strings_and_version(lib):
    assert lib.hsa_status_string(0) == b"HSA_OK"
    assert lib.hsa_status_string(4) == b"HSA_ERR_DEVICE_BOUNDS"
    assert lib.hsa_version() >= 100


def test_workspace_sizes(lib):
    small = _lib.hsa_topk_workspace_size(1, 10, 4)
    big = _lib.hsa_topk_workspace_size(64, 64 * 262144, 512)
    assert 256 < small < big
    assert big >= 8 * 64 * 262144  # candidate buffer covers every score
    assert _lib.hsa_topk_workspace_size(0, 10, 4) == 0


def _rc(fn, *args):
    return getattr(_lib.load(), fn)(*args)


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)        # never dereferenced: validation fails first
    ws = P(0x10000)
    # top-k: k <= 0, k too large, null offsets, misaligned workspace, short workspace
    assert _rc("hsa_topk", fake, fake, 1, 10, 0, fake, None, ws, 1 << 20, None) == 1
    assert _rc("hsa_topk", fake, fake, 1, 10, 4096, fake, None, ws, 1 << 20, None) == 2
    assert _rc("hsa_topk", fake, None, 1, 10, 4, fake, None, ws, 1 << 20, None) == 1
    assert _rc("hsa_topk", fake, fake, 1, 10, 4, fake, None, P(0x10010), 1 << 20, None) == 6
    assert _rc("hsa_topk", fake, fake, 1, 10, 4, fake, None, ws, 16, None) == 6
    assert _rc("hsa_topk", fake, fake, 0, 10, 4, fake, None, ws, 1 << 20, None) == 1
    # compressor: channels not a multiple of 8, r out of range, bad dtype, misaligned
    assert _rc("hsa_compress", fake, fake, fake, 1, 8, 12, 4, fake, 1, None) == 2
    assert _rc("hsa_compress", fake, fake, fake, 1, 8, 16, 0, fake, 1, None) == 2
    assert _rc("hsa_compress", fake, fake, fake, 1, 8, 16, 4, fake, 9, None) == 1
    assert _rc("hsa_compress", P(0x1002), fake, fake, 1, 8, 16, 4, fake, 1, None) == 1
    assert b"16-byte" in lib.hsa_last_error_detail()
    # empty work is a successful no-op that touches nothing
    assert _rc("hsa_compress", None, None, None, 0, 8, 16, 4, None, 1, None) == 0


def test_layer_desc_binding_matches_header():
    """The ctypes descriptor lists hsa_layer_desc's fields in the header's order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct hsa_layer_desc \{(.*?)\} hsa_layer_desc;", text, re.S).group(1)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "int32_t B, Hq, Dqk, Dv" or "const void* const* stage_events" -> field names
        head, *rest = [d.strip() for d in decl.split(",")]
        names.append(re.findall(r"[A-Za-z_][A-Za-z0-9_]*", head)[-1])
        names.extend(rest)
    assert [f[0] for f in _lib.LayerDesc._fields_] == names
