"""Plain CPU oracle for the decode-time hybrid sparse-attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product (the
CUDA library and its binding) never calls it and has no CPU fallback.

The arithmetic lives in ``hsa_oracle.cpp`` (plain C++, double precision, no
CUDA headers, no code shared with the GPU path); this module only compiles it,
marshals numpy arrays into it, and composes the four stages into one decode
layer step the way the pages order them (append -> compress on block
completion -> indexer -> top-k -> attention).

Sources (cited by title and section):
  [KD] kerneldigest.dev, "DeepSeek-V4: optimización de inferencia y RL para
       modelos con atención híbrida y FP4"
  [LH] lehuy.net, "DeepSeek-V4: SGLang và Miles mang đến hỗ trợ Day-0 ..."
  [WK] AI-KOL wiki, "与 SGLang 团队聊 DeepSeek V4:混合注意力的推理与 RL 训练适配"

Arrays of bfloat16 values are passed as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hsa_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

C4, C128 = 4, 128


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (no CUDA involved)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_hardware_threads.restype = ctypes.c_int
            lib.oracle_compress.argtypes = [P, P, P, I64, I64, I64, I64, P, ctypes.c_int]
            lib.oracle_compress_overlap.argtypes = [P, P, P, I64, I64, I64, I64, P, ctypes.c_int]
            lib.oracle_indexer_scores.argtypes = [P, P, P, P, I64, I64, I64, P, ctypes.c_int]
            lib.oracle_topk.argtypes = [P, P, I64, I64, P, P, ctypes.c_int]
            lib.oracle_decode_attn.argtypes = [P, P, P, I64, P, P, P, I64, I64, I64, I64, I64,
                                               ctypes.c_double, P, P, ctypes.c_int]
            lib.oracle_float_to_bf16.argtypes = [P, I64, P]
            lib.oracle_e4m3_to_double.argtypes = [P, I64, P]
            lib.oracle_float_to_e4m3.argtypes = [P, I64, P]
            lib.oracle_quantize_e4m3.argtypes = [P, I64, I64, P, P, ctypes.c_int]
            lib.oracle_indexer_scores_e4m3.argtypes = [P, P, P, P, P, I64, I64, I64, P,
                                                       ctypes.c_int]
            lib.oracle_bf16_to_double.argtypes = [P, I64, P]
            for f in ("oracle_compress", "oracle_compress_overlap", "oracle_indexer_scores", "oracle_topk",
                      "oracle_decode_attn", "oracle_quantize_e4m3",
                      "oracle_indexer_scores_e4m3"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def hardware_threads() -> int:
    return _load().oracle_hardware_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: status {rc}")


def float_to_bf16(x) -> np.ndarray:
    """binary32 -> bfloat16 bits, round to nearest even (the oracle's own rounding)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_float_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_double(x) -> np.ndarray:
    x = _c(x, np.uint16)
    out = np.empty(x.shape, np.float64)
    _load().oracle_bf16_to_double(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_to_double(codes) -> np.ndarray:
    """FP8 E4M3 codes (uint8) -> their values (the format definition; NaN for s.1111.111)."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().oracle_e4m3_to_double(_ptr(codes), codes.size, _ptr(out))
    return out


def float_to_e4m3(x) -> np.ndarray:
    """binary32 -> E4M3 codes: nearest, ties to the even code, saturating at +-448."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().oracle_float_to_e4m3(_ptr(x), x.size, _ptr(out))
    return out


def quantize_e4m3(x, threads: int = 1):
    """Per-row E4M3 quantization: (codes uint8 [rows, C], scales float32 [rows]).

    scale = amax / 448 and code = e4m3(x * (448 / amax)), each step in binary32;
    a zero row gets scale 0.  The library's FP8 storage of the indexer-key pool.
    """
    x = _c(x, np.float32)
    rows, C = x.shape
    codes = np.empty((rows, C), np.uint8)
    scales = np.empty(rows, np.float32)
    _check(_load().oracle_quantize_e4m3(_ptr(x), rows, C, _ptr(codes), _ptr(scales), threads),
           "quantize_e4m3")
    return codes, scales


def dequantize_e4m3(codes, scales) -> np.ndarray:
    """scale[j] * value(code[j, d]) in float64."""
    return e4m3_to_double(codes) * np.asarray(scales, np.float64)[:, None]


def indexer_scores_e4m3(iq, w, keys, kscale, offsets, threads: int = 1) -> np.ndarray:
    """Indexer scores over an E4M3 key pool: the score formula on the dequantized
    keys and on the query rows quantized the same way (per (b, h) row).

    iq: uint16 [B, Hi, Di]; w: float32 [B, Hi]; keys: uint8 [sum N, Di];
    kscale: float32 [sum N]; offsets: int64 [B+1].  Returns float64 [sum N].
    """
    iq, w, keys, kscale, offsets = (_c(iq, np.uint16), _c(w, np.float32), _c(keys, np.uint8),
                                    _c(kscale, np.float32), _c(offsets, np.int64))
    B, Hi, Di = iq.shape
    assert keys.ndim == 2 and keys.shape[1] == Di and kscale.shape == (keys.shape[0],)
    out = np.empty(keys.shape[0], np.float64)
    _check(_load().oracle_indexer_scores_e4m3(_ptr(iq), _ptr(w), _ptr(keys), _ptr(kscale),
                                              _ptr(offsets), B, Hi, Di, _ptr(out), threads),
           "indexer_scores_e4m3")
    return out


def compress(kv, z, b, r: int, threads: int = 1) -> np.ndarray:
    """Flash Compressor (one block of r tokens -> one row, per-channel softmax gate).

    kv, z: uint16 (bf16) [S, T, C]; b: float32 [r, C].  Returns float64 [S, T//r, C].
    [KD] §Arquitectura del Sistema (Flash Compressor); [WK] 推理侧优化 (Kernel fusion).
    """
    kv, z, b = _c(kv, np.uint16), _c(z, np.uint16), _c(b, np.float32)
    S, T, C = kv.shape
    assert z.shape == kv.shape and b.shape == (r, C)
    out = np.empty((S, T // r, C), np.float64)
    _check(_load().oracle_compress(_ptr(kv), _ptr(z), _ptr(b), S, T, C, r, _ptr(out), threads),
           "compress")
    return out


def compress_overlap(kv, z, b, r: int, threads: int = 1) -> np.ndarray:
    """C4 overlap transform: entry n over the 2r-token window of blocks n-1 and n
    (entry 0 over block 0 alone), per-channel softmax gate with a bias b per
    window position.

    kv, z: uint16 (bf16) [S, T, C]; b: float32 [2r, C].  Returns float64 [S, T//r, C].
    [WK] RL 训练侧 ① (C4 overlap transform).
    """
    kv, z, b = _c(kv, np.uint16), _c(z, np.uint16), _c(b, np.float32)
    S, T, C = kv.shape
    assert z.shape == kv.shape and b.shape == (2 * r, C)
    out = np.empty((S, T // r, C), np.float64)
    _check(_load().oracle_compress_overlap(_ptr(kv), _ptr(z), _ptr(b), S, T, C, r, _ptr(out),
                                           threads), "compress_overlap")
    return out


def indexer_scores(iq, w, keys, offsets, threads: int = 1) -> np.ndarray:
    """s[j] = sum_h w_h * relu(q_h . k_j) over each sequence's compressed entries.

    iq: uint16 [B, Hi, Di]; w: float32 [B, Hi]; keys: uint16 [sum N, Di];
    offsets: int64 [B+1].  Returns float64 [sum N].  [KD] flow step 6 (indexer).
    """
    iq, w, keys, offsets = (_c(iq, np.uint16), _c(w, np.float32), _c(keys, np.uint16),
                            _c(offsets, np.int64))
    B, Hi, Di = iq.shape
    assert keys.ndim == 2 and keys.shape[1] == Di and offsets.shape == (B + 1,)
    out = np.empty(keys.shape[0], np.float64)
    _check(_load().oracle_indexer_scores(_ptr(iq), _ptr(w), _ptr(keys), _ptr(offsets), B, Hi, Di,
                                         _ptr(out), threads), "indexer_scores")
    return out


def topk(scores, offsets, k: int, threads: int = 1):
    """Top-k by (value desc, index asc) per row; -1 / -inf padding.  Returns (idx, vals).

    scores: float32 [sum N]; offsets: int64 [B+1].  [KD] §Arquitectura (Lightning TopK).
    """
    scores, offsets = _c(scores, np.float32), _c(offsets, np.int64)
    B = offsets.shape[0] - 1
    idx = np.empty((B, k), np.int32)
    vals = np.empty((B, k), np.float32)
    _check(_load().oracle_topk(_ptr(scores), _ptr(offsets), B, k, _ptr(idx), _ptr(vals), threads),
           "topk")
    return idx, vals


def decode_attn(q, swa, seq_len, W: int, extra, extra_offsets, extra_idx, scale: float,
                Dv: int, threads: int = 1):
    """One softmax over the SWA window plus the listed (or all) compressed rows.

    q: uint16 [B, Hq, Dqk]; swa: uint16 [B, W, Dqk] ring (slot = pos mod W);
    seq_len: int32 [B]; extra: uint16 [sum N, Dqk] or None; extra_offsets: int64
    [B+1] or None; extra_idx: int32 [B, k] or None (dense).  Returns
    (out float64 [B, Hq, Dv], lse float64 [B, Hq]).  [KD] flow step 5.
    """
    q, swa, seq_len = _c(q, np.uint16), _c(swa, np.uint16), _c(seq_len, np.int32)
    B, Hq, Dqk = q.shape
    assert swa.shape == (B, W, Dqk)
    if extra is not None:
        extra, extra_offsets = _c(extra, np.uint16), _c(extra_offsets, np.int64)
    k = 0
    if extra_idx is not None:
        extra_idx = _c(extra_idx, np.int32)
        k = extra_idx.shape[1]
    out = np.empty((B, Hq, Dv), np.float64)
    lse = np.empty((B, Hq), np.float64)
    _check(_load().oracle_decode_attn(_ptr(q), _ptr(swa), _ptr(seq_len), W, _ptr(extra),
                                      _ptr(extra_offsets), _ptr(extra_idx), k, B, Hq, Dqk, Dv,
                                      float(scale), _ptr(out), _ptr(lse), threads),
           "decode_attn")
    return out, lse


def compact(pool, pool_offsets, counts):
    """Rows [off_b, off_b + counts[b]) of a capacity-laid-out pool, concatenated."""
    parts = [pool[int(pool_offsets[b]):int(pool_offsets[b]) + int(counts[b])]
             for b in range(len(counts))]
    offs = np.zeros(len(counts) + 1, np.int64)
    offs[1:] = np.cumsum([int(c) for c in counts])
    width = pool.shape[1]
    rows = np.concatenate(parts, axis=0) if parts else np.zeros((0, width), pool.dtype)
    return rows.reshape(-1, width), offs


def _window_ring(swa, L, W):
    """The last W positions of each sequence (positions [max(0, L-W), L)) from a
    ring of any size Wr >= W (slot = position mod Wr), re-laid as a ring of W
    slots (slot = position mod W): data movement only."""
    B, Wr, D = swa.shape
    out = np.zeros((B, W, D), swa.dtype)
    for b in range(B):
        for p in range(max(0, int(L[b]) - W), int(L[b])):
            out[b, p % W] = swa[b, p % Wr]
    return out


def layer_decode(st: dict, threads: int = 1) -> dict:
    """One decode step of one hybrid layer, composed from the four stages.

    The step order follows the data dependence the pages describe ([WK] 核心观点:
    compress once a 4- / 128-token block is complete, C4 picks its top-k entries
    and then attends them; [KD] flow steps 3, 5 and 6):

      a1 append the new tokens' rows, in order, into the SWA ring (slot p mod
         Wr) and the in-flight block rings (slot p mod r), p = L_in + t;
      a2 when a token completes a block ((p + 1) mod r == 0), compress the block
         into pool row (p + 1)/r - 1 (compressor output rounded fp64 -> fp32
         -> bf16, as stored; with an E4M3 key pool (``st["key_fp8"]``) the
         indexer key is rounded to fp32 and quantized per row into
         ``key_pool`` codes and ``key_scale``);
      a3 (C4) for each query token t (length L_t = L_in + t + 1), indexer
         scores over its L_t/4 entries, rounded to fp32;
      a4 (C4) top-k of those scores;
      a5 attention of token t over its window (positions [L_t - W, L_t)) and
         its selected (C4) or all (C128) rows.

    ``st["T"]`` (default 1) query tokens per sequence — T = 2 is one step of
    speculative decoding with a one-layer multi-token-prediction head ([LH]
    §Tích hợp Kernel và Giải mã suy đoán): the current token and a draft
    token, verified together.  Token t sees exactly what it would see had the
    tokens been decoded one per step (its own and earlier positions only); the
    window ring holds Wr = W + T - 1 rows so that the first token's oldest
    window row survives the later appends.  With T > 1 the per-token inputs
    carry a token axis after the batch axis (q [B, T, Hq, Dqk], kv_new
    [B, T, Dqk], iq [B, T, Hi, Di], w [B, T, Hi], ...) and so do the outputs.

    ``st`` holds numpy arrays (see the keys read below); the rings and pools in
    it are updated in place.  Returns the stage outputs.
    """
    kind, r = st["kind"], st["ratio"]
    T = int(st.get("T", 1))
    B = st["seq_len_in"].shape[0]
    Wr = st["swa"].shape[1]
    W = int(st.get("W", Wr - (T - 1)))
    assert Wr >= W + T - 1, "the window ring needs W + T - 1 rows"
    Lin = st["seq_len_in"].astype(np.int64)
    L = Lin + T
    Dv = st["Dv"]

    def tok(name, t):
        a = st[name]
        return a if T == 1 else a[:, t]

    out = {"seq_len_out": L.astype(np.int32)}
    offs = st["pool_offsets"]
    for t in range(T):
        for b in range(B):
            p = int(Lin[b]) + t
            st["swa"][b, p % Wr] = tok("kv_new", t)[b]
            st["kv_ring"][b, p % r] = tok("kv_new", t)[b]
            st["z_ring"][b, p % r] = tok("z_new", t)[b]
            if kind == C4:
                st["ik_ring"][b, p % r] = tok("ik_new", t)[b]
                st["iz_ring"][b, p % r] = tok("iz_new", t)[b]
            if (p + 1) % r != 0:
                continue
            n = (p + 1) // r - 1
            assert offs[b] + n < offs[b + 1], "pool capacity exceeded"
            c = compress(st["kv_ring"][b:b + 1], st["z_ring"][b:b + 1], st["b_kv"], r, threads)
            st["kv_pool"][offs[b] + n] = float_to_bf16(c.astype(np.float32)).reshape(-1)
            if kind == C4:
                ck = compress(st["ik_ring"][b:b + 1], st["iz_ring"][b:b + 1], st["b_ik"], r,
                              threads)
                if st.get("key_fp8"):
                    codes, sc = quantize_e4m3(ck.astype(np.float32).reshape(1, -1))
                    st["key_pool"][offs[b] + n] = codes[0]
                    st["key_scale"][offs[b] + n] = sc[0]
                else:
                    st["key_pool"][offs[b] + n] = float_to_bf16(ck.astype(np.float32)).reshape(-1)
    res = []
    for t in range(T):
        Lt = Lin + t + 1
        counts = Lt // r
        kv_rows, kv_offs = compact(st["kv_pool"], offs, counts)
        rt = {}
        idx = None
        if kind == C4:
            key_rows, key_offs = compact(st["key_pool"], offs, counts)
            if st.get("key_fp8"):
                ksc, _ = compact(st["key_scale"].reshape(-1, 1), offs, counts)
                s64 = indexer_scores_e4m3(tok("iq", t), tok("w", t), key_rows, ksc.reshape(-1),
                                          key_offs, threads)
            else:
                s64 = indexer_scores(tok("iq", t), tok("w", t), key_rows, key_offs, threads)
            s32 = s64.astype(np.float32)
            idx, vals = topk(s32, key_offs, st["k"], threads)
            rt.update(scores64=s64, scores=s32, score_offsets=key_offs, idx=idx, vals=vals)
        ring = st["swa"] if Wr == W else _window_ring(st["swa"], Lt, W)
        o, lse = decode_attn(tok("q", t), ring, Lt.astype(np.int32), W, kv_rows, kv_offs, idx,
                             st["scale"], Dv, threads)
        rt.update(out=o, lse=lse)
        res.append(rt)
    if T == 1:
        out.update(res[0])
    else:
        out["tokens"] = res
        for key in ("out", "lse", "idx"):
            if key in res[0]:
                out[key] = np.stack([rt[key] for rt in res], axis=1)
    return out
