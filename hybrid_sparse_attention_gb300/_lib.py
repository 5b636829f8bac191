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
    "hsa_compress_overlap": (I32, [P, P, P, I64, I64, I64, I64, P, I32, P]),
    "hsa_indexer_scores_workspace_size": (SZ, []),
    "hsa_indexer_scores": (I32, [P, P, P, P, I64, I64, I64, I64, P, P, SZ, P]),
    "hsa_decode_attn_workspace_size": (SZ, [I64, I64, I64, I64, I64, I64]),
    "hsa_decode_attn": (I32, [P, P, P, I64, P, P, I64, P, I64, I64, I64, I64, I64, I64,
                              ctypes.c_float, P, I32, P, P, SZ, P]),
    "hsa_topk_workspace_size": (SZ, [I64, I64, I64]),
    "hsa_topk": (I32, [P, P, I64, I64, I64, P, P, P, SZ, P]),
    "hsa_topk_noalloc": (I32, [P, P, I64, I64, I64, P, P, P]),
    "hsa_quantize_e4m3": (I32, [P, I64, I64, P, P, P]),
    "hsa_set_wait_limit": (I32, [ctypes.c_uint64, ctypes.c_uint32]),
    "hsa_indexer_scores_e4m3": (I32, [P, P, P, P, P, I64, I64, I64, I64, P, P, SZ, P]),
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


def hsa_compress_overlap(kv, z, b, r: int, out=None, out_dtype=torch.bfloat16, stream=None):
    """C4 overlap transform: kv, z bf16 [S, T, C]; b fp32 [2r, C] -> out [S, T//r, C]
    (entry n over the window of blocks n-1 and n)."""
    S, T, C = kv.shape
    if out is None:
        out = torch.empty(S, T // r, C, dtype=out_dtype, device=kv.device)
    code = {torch.float32: HSA_F32, torch.bfloat16: HSA_BF16}[out.dtype]
    _call("hsa_compress_overlap", _dev(kv, torch.bfloat16, "kv"), _dev(z, torch.bfloat16, "z"),
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


def hsa_quantize_e4m3(x, codes=None, scales=None, stream=None):
    """Per-row E4M3 quantization: x fp32 [rows, C] -> (codes uint8 [rows, C],
    scales fp32 [rows]), scale = amax / 448, code = e4m3(x * 448 / amax)."""
    rows, C = x.shape
    if codes is None:
        codes = torch.empty(rows, C, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    _call("hsa_quantize_e4m3", _dev(x, torch.float32, "x"), rows, C,
          _dev(codes, torch.uint8, "codes"), _dev(scales, torch.float32, "scales"),
          _stream(stream))
    return codes, scales


def hsa_indexer_scores_e4m3(iq, w, keys, key_scales, offsets, scores=None, ws=None, stream=None):
    """Indexer scores over an E4M3 key pool: iq bf16 [B,Hi,128] (quantized per row
    in the kernel), w fp32 [B,Hi], keys uint8 [total,128], key_scales fp32
    [total], offsets int64 [B+1] (device) -> scores fp32 [total]."""
    B, Hi, Di = iq.shape
    total = keys.shape[0]
    if scores is None:
        scores = torch.zeros(total, dtype=torch.float32, device=keys.device)
    if ws is None:
        ws = workspace(hsa_indexer_scores_workspace_size(), keys.device)
    _call("hsa_indexer_scores_e4m3", _dev(iq, torch.bfloat16, "iq"), _dev(w, torch.float32, "w"),
          _dev(keys, torch.uint8, "keys"), _dev(key_scales, torch.float32, "key_scales"),
          _dev(offsets, torch.int64, "offsets"), B, Hi, Di, total,
          _dev(scores, torch.float32, "scores"), _dev(ws, torch.uint8, "ws"), ws.numel(),
          _stream(stream))
    return scores


def hsa_set_wait_limit(nanos: int = 0, polls: int = 0) -> None:
    """Bound of the indexer kernels' pipeline waits for later launches (0: default)."""
    _call("hsa_set_wait_limit", int(nanos), int(polls))


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


def hsa_topk_noalloc(scores, offsets, k: int, idx=None, vals=None, with_vals=True, stream=None):
    """Top-k without a workspace (scratch in the library's static device array).
    Output tensors are allocated here when not given; the C call allocates nothing."""
    B = offsets.numel() - 1
    if idx is None:
        idx = torch.empty(B, k, dtype=torch.int32, device=scores.device)
    if vals is None and with_vals:
        vals = torch.empty(B, k, dtype=torch.float32, device=scores.device)
    _call("hsa_topk_noalloc", _dev(scores, torch.float32, "scores"),
          _dev(offsets, torch.int64, "offsets"), B, scores.numel(), k,
          _dev(idx, torch.int32, "idx"), _dev(vals, torch.float32, "vals", True), _stream(stream))
    return idx, vals


class LayerDesc(ctypes.Structure):
    """Mirror of hsa_layer_desc (include/hsa.h)."""
    _fields_ = [
        ("kind", ctypes.c_int32), ("B", ctypes.c_int32), ("Hq", ctypes.c_int32),
        ("Dqk", ctypes.c_int32), ("Dv", ctypes.c_int32), ("Hi", ctypes.c_int32),
        ("Di", ctypes.c_int32), ("W", ctypes.c_int32), ("k", ctypes.c_int32),
        ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int32),
        ("pool_total_rows", ctypes.c_int64), ("max_pool_rows", ctypes.c_int64),
        ("seq_len_in", P), ("seq_len_out", P), ("pool_offsets", P),
        ("kv_new", P), ("z_new", P), ("b_kv", P), ("ik_new", P), ("iz_new", P), ("b_ik", P),
        ("swa", P), ("kv_ring", P), ("z_ring", P), ("ik_ring", P), ("iz_ring", P),
        ("kv_pool", P), ("key_pool", P), ("q", P), ("iq", P), ("w", P),
        ("out", P), ("lse", P), ("topk_idx", P), ("scores", P), ("stage_events", P),
        ("q_ready_event", P), ("key_fp8", ctypes.c_int32), ("key_scale", P),
        ("T", ctypes.c_int32),
    ]


SIGNATURES["hsa_layer_decode_workspace_size"] = (SZ, [ctypes.POINTER(LayerDesc)])
SIGNATURES["hsa_layer_decode_launches"] = (I32, [ctypes.POINTER(LayerDesc)])
SIGNATURES["hsa_layer_decode"] = (I32, [ctypes.POINTER(LayerDesc), P, SZ, P])


def layer_desc(st, out, lse=None, seq_len_out=None, topk_idx=None, scores=None,
               max_pool_rows=None, stage_events=None, q_ready_event=None) -> LayerDesc:
    """Descriptor for one decode step over a synth.LayerState-like object whose
    tensors live on the GPU (argument marshalling only)."""
    sh = st.shape
    c4 = st.kind == HSA_LAYER_C4
    d = LayerDesc()
    d.kind = st.kind
    d.B = st.seq_len_in.numel()
    d.Hq, d.Dqk, d.Dv = sh.Hq, sh.Dqk, sh.Dv
    d.Hi, d.Di = (sh.Hi, sh.Di) if c4 else (0, 0)
    d.W, d.k = sh.W, (sh.k if c4 else 0)
    d.scale = sh.scale
    d.T = getattr(st, "T", 1)
    d.out_dtype = {torch.float32: HSA_F32, torch.bfloat16: HSA_BF16}[out.dtype]
    d.pool_total_rows = st.kv_pool.shape[0]
    if max_pool_rows is None:   # the largest pool capacity bounds every live count
        max_pool_rows = int((st.pool_offsets[1:] - st.pool_offsets[:-1]).max())
    d.max_pool_rows = max_pool_rows
    d.seq_len_in = _dev(st.seq_len_in, torch.int32, "seq_len_in")
    d.seq_len_out = _dev(st.seq_len_in if seq_len_out is None else seq_len_out, torch.int32,
                         "seq_len_out")
    d.pool_offsets = _dev(st.pool_offsets, torch.int64, "pool_offsets")
    d.kv_new = _dev(st.kv_new, torch.bfloat16, "kv_new")
    d.z_new = _dev(st.z_new, torch.bfloat16, "z_new")
    d.b_kv = _dev(st.b_kv, torch.float32, "b_kv")
    d.swa = _dev(st.swa, torch.bfloat16, "swa")
    d.kv_ring = _dev(st.kv_ring, torch.bfloat16, "kv_ring")
    d.z_ring = _dev(st.z_ring, torch.bfloat16, "z_ring")
    d.kv_pool = _dev(st.kv_pool, torch.bfloat16, "kv_pool")
    d.q = _dev(st.q, torch.bfloat16, "q")
    if c4:
        d.ik_new = _dev(st.ik_new, torch.bfloat16, "ik_new")
        d.iz_new = _dev(st.iz_new, torch.bfloat16, "iz_new")
        d.b_ik = _dev(st.b_ik, torch.float32, "b_ik")
        d.ik_ring = _dev(st.ik_ring, torch.bfloat16, "ik_ring")
        d.iz_ring = _dev(st.iz_ring, torch.bfloat16, "iz_ring")
        # an E4M3 key pool: uint8 codes with one fp32 scale per row
        key_scale = getattr(st, "key_scale", None)
        d.key_pool = _dev(st.key_pool, torch.bfloat16 if key_scale is None else torch.uint8,
                          "key_pool")
        if key_scale is not None:
            d.key_fp8 = 1
            d.key_scale = _dev(key_scale, torch.float32, "key_scale")
        d.iq = _dev(st.iq, torch.bfloat16, "iq")
        d.w = _dev(st.w, torch.float32, "w")
        d.topk_idx = _dev(topk_idx, torch.int32, "topk_idx", True)
        d.scores = _dev(scores, torch.float32, "scores", True)
    d.out = _dev(out, out.dtype, "out")
    d.lse = _dev(lse, torch.float32, "lse", True)
    if stage_events is not None:
        # keep the handle array alive as long as the descriptor
        d._events = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(h) for h in stage_events])
        d.stage_events = ctypes.cast(d._events, ctypes.c_void_p)
    if q_ready_event is not None:   # a cudaEvent_t handle (torch.cuda.Event.cuda_event)
        d.q_ready_event = q_ready_event
    # the descriptor holds raw device pointers: keep every tensor behind them
    # alive as long as it is (a temporary passed here would otherwise be freed
    # and its memory handed to another tensor while the library still writes it)
    d._keep = (st, out, lse, seq_len_out, topk_idx, scores)
    return d


def hsa_layer_decode_workspace_size(desc: LayerDesc) -> int:
    return int(load().hsa_layer_decode_workspace_size(ctypes.byref(desc)))


def hsa_layer_decode_launches(desc: LayerDesc) -> int:
    """Kernel launches one hsa_layer_decode call with this descriptor makes."""
    return int(load().hsa_layer_decode_launches(ctypes.byref(desc)))


def hsa_layer_decode(desc: LayerDesc, ws=None, stream=None):
    """One decode step of one hybrid layer (append, compress, [score, top-k], attend)."""
    if ws is None:
        ws = workspace(hsa_layer_decode_workspace_size(desc))
    _call("hsa_layer_decode", ctypes.byref(desc), _dev(ws, torch.uint8, "ws"), ws.numel(),
          _stream(stream))
    return ws
