"""Thin Python binding of libhsa.so (the C ABI in include/hsa.h).

Argument marshalling only: each function takes torch tensors, checks dtype /
device / contiguity, passes their device pointers and the current CUDA stream
to the C entry point of the same name, and raises HsaError on a non-OK status.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback.  If the library has not been built, loading fails
loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

HSA_F32, HSA_BF16 = 0, 1
HSA_LAYER_C4, HSA_LAYER_C128 = 4, 128
STATUS = {0: "HSA_OK", 1: "HSA_ERR_INVALID_ARG", 2: "HSA_ERR_UNSUPPORTED", 3: "HSA_ERR_CUDA",
          4: "HSA_ERR_DEVICE_BOUNDS", 5: "HSA_ERR_TIMEOUT", 6: "HSA_ERR_WORKSPACE",
          7: "HSA_ERR_NAN"}

P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/hsa.h
SIGNATURES = {
    "hsa_status_string": (ctypes.c_char_p, [I32]),
    "hsa_last_error_detail": (ctypes.c_char_p, []),
    "hsa_version": (I32, []),
    "hsa_workspace_status": (I32, [P, P, P]),
    "hsa_compress": (I32, [P, P, P, I64, I64, I64, I64, P, I32, P]),
    "hsa_indexer_scores_workspace_size": (SZ, []),
    "hsa_indexer_scores": (I32, [P, P, P, P, I64, I64, I64, I64, P, P, SZ, P]),
    "hsa_decode_attn_workspace_size": (SZ, [I64, I64, I64, I64, I64, I64]),
    "hsa_decode_attn": (I32, [P, P, P, I64, P, P, I64, P, I64, I64, I64, I64, I64, I64,
                              ctypes.c_float, P, I32, P, P, SZ, P]),
    "hsa_topk_workspace_size": (SZ, [I64, I64, I64]),
    "hsa_topk": (I32, [P, P, I64, I64, I64, P, P, P, SZ, P]),
}


class HsaError(RuntimeError):
    def __init__(self, code: int, fn: str, detail: str):
        self.code = code
        super().__init__(f"{fn}: {STATUS.get(code, code)}: {detail}")


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libhsa.so (optionally building it first).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise ImportError(f"libhsa.so not built ({path}); run __graft_entry__.build()")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _lib = lib
    return _lib


def _call(name: str, *args) -> None:
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != 0:
        raise HsaError(rc, name, lib.hsa_last_error_detail().decode())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled, 256-byte aligned device workspace of at least nbytes."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def hsa_workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Reads and clears the sticky device status bits of a workspace (synchronises)."""
    bits = ctypes.c_uint32(0)
    lib = load()
    rc = lib.hsa_workspace_status(ctypes.c_void_p(ws.data_ptr()), _stream(stream),
                                  ctypes.byref(bits))
    if rc not in (0, 4, 5, 7):
        raise HsaError(rc, "hsa_workspace_status", lib.hsa_last_error_detail().decode())
    return bits.value


def hsa_compress(kv, z, b, r: int, out=None, out_dtype=torch.bfloat16, stream=None):
    """Flash Compressor: kv, z bf16 [S, T, C]; b fp32 [r, C] -> out [S, T//r, C]."""
    S, T, C = kv.shape
    if out is None:
        out = torch.empty(S, T // r, C, dtype=out_dtype, device=kv.device)
    code = {torch.float32: HSA_F32, torch.bfloat16: HSA_BF16}[out.dtype]
    _call("hsa_compress", _dev(kv, torch.bfloat16, "kv"), _dev(z, torch.bfloat16, "z"),
          _dev(b, torch.float32, "b"), S, T, C, r, _dev(out, out.dtype, "out"), code,
          _stream(stream))
    return out


def hsa_indexer_scores_workspace_size() -> int:
    return int(load().hsa_indexer_scores_workspace_size())


def hsa_indexer_scores(iq, w, keys, offsets, scores=None, ws=None, stream=None):
    """s[j] = sum_h w[b,h] relu(iq[b,h] . keys[j]): iq bf16 [B,Hi,Di], w fp32 [B,Hi],
    keys bf16 [total, Di], offsets int64 [B+1] (device) -> scores fp32 [total]."""
    B, Hi, Di = iq.shape
    total = keys.shape[0]
    if scores is None:
        scores = torch.zeros(total, dtype=torch.float32, device=keys.device)
    if ws is None:
        ws = workspace(hsa_indexer_scores_workspace_size(), keys.device)
    _call("hsa_indexer_scores", _dev(iq, torch.bfloat16, "iq"), _dev(w, torch.float32, "w"),
          _dev(keys, torch.bfloat16, "keys"), _dev(offsets, torch.int64, "offsets"), B, Hi, Di,
          total, _dev(scores, torch.float32, "scores"), _dev(ws, torch.uint8, "ws"), ws.numel(),
          _stream(stream))
    return scores


def hsa_topk_workspace_size(B: int, total_rows: int, k: int) -> int:
    return int(load().hsa_topk_workspace_size(B, total_rows, k))


def hsa_topk(scores, offsets, k: int, idx=None, vals=None, ws=None, with_vals=True, stream=None):
    """Top-k per ragged row: scores fp32 [sum N], offsets int64 [B+1] (device).
    Returns (idx int32 [B, k], vals fp32 [B, k] or None)."""
    B = offsets.numel() - 1
    total = scores.numel()
    if idx is None:
        idx = torch.empty(B, k, dtype=torch.int32, device=scores.device)
    if vals is None and with_vals:
        vals = torch.empty(B, k, dtype=torch.float32, device=scores.device)
    need = hsa_topk_workspace_size(B, total, k)
    if ws is None:
        ws = workspace(need, scores.device)
    _call("hsa_topk", _dev(scores, torch.float32, "scores"), _dev(offsets, torch.int64, "offsets"),
          B, total, k, _dev(idx, torch.int32, "idx"), _dev(vals, torch.float32, "vals", True),
          _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    return idx, vals


def hsa_decode_attn_workspace_size(B, Hq, Dqk, Dv, W, extra_slots) -> int:
    return int(load().hsa_decode_attn_workspace_size(B, Hq, Dqk, Dv, W, extra_slots))


def hsa_decode_attn(q, swa, seq_len, extra=None, extra_offsets=None, extra_idx=None,
                    max_extra_rows=0, scale=None, Dv=None, out=None, out_dtype=torch.bfloat16,
                    lse=None, ws=None, stream=None):
    """Fused SWA + compressed attention for one query token per sequence.

    q bf16 [B, Hq, Dqk]; swa bf16 [B, W, Dqk] ring; seq_len int32 [B]; extra bf16
    [rows, Dqk] with extra_offsets int64 [B+1]; extra_idx int32 [B, k] (sparse) or
    None (dense, N_b <= max_extra_rows).  Returns (out [B, Hq, Dv], lse fp32 [B, Hq])."""
    B, Hq, Dqk = q.shape
    W = swa.shape[1]
    Dv = Dqk if Dv is None else Dv
    scale = (1.0 / Dqk ** 0.5) if scale is None else scale
    k = extra_idx.shape[1] if extra_idx is not None else 0
    rows = extra.shape[0] if extra is not None else 0
    if out is None:
        out = torch.empty(B, Hq, Dv, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    slots = k if extra_idx is not None else max_extra_rows
    need = hsa_decode_attn_workspace_size(B, Hq, Dqk, Dv, W, slots)
    if ws is None:
        ws = workspace(need, q.device)
    code = {torch.float32: HSA_F32, torch.bfloat16: HSA_BF16}[out.dtype]
    _call("hsa_decode_attn", _dev(q, torch.bfloat16, "q"), _dev(swa, torch.bfloat16, "swa"),
          _dev(seq_len, torch.int32, "seq_len"), W, _dev(extra, torch.bfloat16, "extra", True),
          _dev(extra_offsets, torch.int64, "extra_offsets", True), rows,
          _dev(extra_idx, torch.int32, "extra_idx", True), k, max_extra_rows, B, Hq, Dqk, Dv,
          float(scale), _dev(out, out.dtype, "out"), code, _dev(lse, torch.float32, "lse", True),
          _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    return out, lse
