"""Seeded synthetic inputs for the decode-time hybrid sparse-attention path.

This module only draws numbers and arranges them into the shapes, value
distributions and structure of the workloads (ragged context lengths, tie
patterns, pool layouts).  It holds none of the method's arithmetic, and both
the CUDA path and the CPU oracle consume what it produces.

Generator (counter based, so any slice can be produced independently):
  * draw i of stream s is splitmix64 applied to  seed_s + (i + 1) * 0x9E3779B97F4A7C15,
    seed_s = splitmix64(seed ^ crc32(stream name));
  * a uniform in (0, 1) takes 24 bits:  (bits + 0.5) * 2**-24;
  * normals come in pairs from one 64-bit draw by Box-Muller in float64
    (top 24 bits -> radius, next 24 bits -> angle), then rounded to float32;
  * bf16 values are the float32 values rounded to nearest even by torch.
The integer part is exact on every device.  The Box-Muller transcendental
functions may differ in the last float64 bit between a CPU and a GPU, so a
parity case draws its inputs once, on one device, and hands the same bits to
both sides.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 24


def _s64(c: int) -> int:
    c &= (1 << 64) - 1
    return c - (1 << 64) if c >= (1 << 63) else c


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor holding uint64 bits."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(_M1)
    z = (z ^ _srl(z, 27)) * _s64(_M2)
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * _M1) & m
    z = ((z ^ (z >> 27)) * _M2) & m
    return z ^ (z >> 31)


def stream_seed(seed: int, name: str) -> int:
    return _mix_int((seed ^ zlib.crc32(name.encode())) + _GOLDEN)


def bits(seed: int, name: str, n: int, device="cpu", start: int = 0) -> torch.Tensor:
    """n raw 64-bit draws (int64 tensor) of stream `name`, draws start..start+n-1."""
    s = stream_seed(seed, name)
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    return _mix(i * _s64(_GOLDEN) + _s64(s))


def uniform(seed: int, name: str, shape, device="cpu") -> torch.Tensor:
    """float32 U(0, 1) from the top 24 bits of each draw."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        u = _srl(bits(seed, name, hi - lo, device, lo), 40).to(torch.float64)
        out[lo:hi] = ((u + 0.5) * 2.0 ** -24).to(torch.float32)
    return out.reshape(shape)


def normal(seed: int, name: str, shape, std: float = 1.0, device="cpu") -> torch.Tensor:
    """float32 N(0, std^2) by Box-Muller, two normals per 64-bit draw."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    per = 2 * _CHUNK
    for lo in range(0, n, per):
        hi = min(n, lo + per)
        m = (hi - lo + 1) // 2
        x = bits(seed, name, m, device, lo // 2)
        u1 = (_srl(x, 40).to(torch.float64) + 0.5) * 2.0 ** -24
        u2 = ((_srl(x, 16) & 0xFFFFFF).to(torch.float64) + 0.5) * 2.0 ** -24
        rad = torch.sqrt(-2.0 * torch.log(u1)) * std
        ang = 2.0 * math.pi * u2
        pair = torch.stack([rad * torch.cos(ang), rad * torch.sin(ang)], dim=1).reshape(-1)
        out[lo:hi] = pair[: hi - lo].to(torch.float32)
    return out.reshape(shape)


def normal_bf16(seed, name, shape, std=1.0, device="cpu") -> torch.Tensor:
    return normal(seed, name, shape, std, device).to(torch.bfloat16)


def randint(seed: int, name: str, n: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """int64 uniform integers in [lo, hi] (inclusive), from the top 32 bits of each draw."""
    x = _srl(bits(seed, name, n, device), 32)
    return lo + (x * (hi - lo + 1)) // (1 << 32)


def permutation(seed: int, name: str, n: int, device="cpu") -> torch.Tensor:
    """A uniform random permutation of range(n): stable argsort of n random keys."""
    return torch.sort(_srl(bits(seed, name, n, device), 1), stable=True).indices


# --------------------------------------------------------------------------
# Workloads (shapes and structure of the pages' / this library's configs)
# --------------------------------------------------------------------------

@dataclass
class LayerShape:
    """Head shapes of one hybrid layer."""
    Hq: int
    Dqk: int
    Dv: int
    Hi: int
    Di: int
    k: int
    W: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dqk)


TINY = LayerShape(Hq=8, Dqk=128, Dv=128, Hi=2, Di=32, k=64, W=64)
FULL = LayerShape(Hq=64, Dqk=576, Dv=512, Hi=8, Di=128, k=512, W=128)

SEED = {"tiny": 0x48534101, "topk": 0x48534102, "compress": 0x48534103,
        "c4layer": 0x48534104, "longctx": 0x48534105}


def topk_scores(seed: int, rows: int, n: int, dup_frac: float = 0.05, device="cpu"):
    """fp32 [rows, n] ~ N(0,1); then per row floor(dup_frac * n) distinct positions,
    chosen uniformly without replacement, are overwritten with the original value
    of a uniformly chosen other position of the same row (forces ties)."""
    x = normal(seed, "topk.scores", (rows, n), device=device)
    m = int(dup_frac * n)
    if m == 0 or n < 2:
        return x
    orig = x.clone()
    for r in range(rows):
        tgt = permutation(seed, f"topk.dup_pos.{r}", n, device)[:m]
        step = randint(seed, f"topk.dup_src.{r}", m, 1, n - 1, device)
        src = (tgt + step) % n
        x[r, tgt] = orig[r, src]
    return x


def pair_ties_at_top(row: torch.Tensor, top: int = 600) -> torch.Tensor:
    """Adversarial tie pattern: the `top` largest values of a row, in sorted
    order, are made equal in pairs (2i+1 takes the value of 2i), so equal values
    straddle every rank near the threshold."""
    row = row.clone()
    order = torch.sort(row, descending=True, stable=True).indices[:top]
    vals = row[order]
    vals[1::2] = vals[0::2][: vals[1::2].numel()]
    row[order] = vals
    return row


def c4_lengths(seed: int, B: int, lo: int = 16384, hi: int = 131072) -> torch.Tensor:
    """Context lengths L_b (tokens after this step's append) ~ U[lo, hi] integers."""
    return randint(seed, "c4layer.L", B, lo, hi).to(torch.int32)


def capacity_offsets(counts, slack: int = 1) -> torch.Tensor:
    """int64 [B+1] start offsets of a capacity-laid-out pool with `counts[b] + slack` rows each."""
    caps = torch.as_tensor(counts, dtype=torch.int64) + slack
    offs = torch.zeros(caps.numel() + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(caps, 0)
    return offs


@dataclass
class LayerState:
    """Tensors of one hybrid layer's decode step (all bf16 unless noted)."""
    kind: int
    ratio: int
    shape: LayerShape
    seq_len_in: torch.Tensor        # int32 [B], tokens before this step
    pool_offsets: torch.Tensor      # int64 [B+1], capacity layout
    swa: torch.Tensor               # [B, W, Dqk]
    kv_ring: torch.Tensor           # [B, r, Dqk]
    z_ring: torch.Tensor            # [B, r, Dqk]
    kv_pool: torch.Tensor           # [cap, Dqk]
    b_kv: torch.Tensor              # fp32 [r, Dqk]
    kv_new: torch.Tensor            # [B, Dqk]
    z_new: torch.Tensor             # [B, Dqk]
    q: torch.Tensor                 # [B, Hq, Dqk]
    ik_ring: torch.Tensor = None    # [B, r, Di]   (C4)
    iz_ring: torch.Tensor = None    # [B, r, Di]   (C4)
    key_pool: torch.Tensor = None   # [cap, Di]    (C4)
    b_ik: torch.Tensor = None       # fp32 [r, Di] (C4)
    ik_new: torch.Tensor = None     # [B, Di]      (C4)
    iz_new: torch.Tensor = None     # [B, Di]      (C4)
    iq: torch.Tensor = None         # [B, Hi, Di]  (C4)
    w: torch.Tensor = None          # fp32 [B, Hi] (C4)
    key_scale: torch.Tensor = None  # fp32 [cap] when key_pool holds E4M3 codes (uint8 [cap, Di])
    T: int = 1                      # query tokens per sequence and step; with T > 1 the
                                    # per-token tensors (q, kv_new, z_new, ik_new, iz_new,
                                    # iq, w) have a token axis after the batch axis and the
                                    # window ring holds W + T - 1 rows
    extra: dict = field(default_factory=dict)

    def tensors(self):
        return {k: v for k, v in self.__dict__.items() if isinstance(v, torch.Tensor)}

    def to(self, device):
        kw = dict(self.__dict__)
        for k, v in self.tensors().items():
            kw[k] = v.to(device)
        return LayerState(**kw)


def raw_token_state(seed: int, kind: int, shape: LayerShape, L: int, device="cpu",
                    slack: int = 1):
    """A single-sequence layer whose history is L-1 raw tokens (kv, z ~ N(0,1);
    indexer raw keys and their gates ~ N(0,1)), plus the new token, positional
    biases b ~ N(0, 0.5^2), q ~ N(0,1), indexer q ~ N(0,1) and w ~ U(0,1).
    The compressed pools are left empty (zero): the caller builds them from the
    raw history with its own compressor; each pool has room for `slack` rows
    beyond L // r.  Returns (state, raw) where raw holds the history tensors."""
    r = kind
    name = "c4" if kind == 4 else "c128"
    D, Di = shape.Dqk, shape.Di
    hist = L - 1
    raw = {"kv": normal_bf16(seed, f"{name}.kv", (1, hist, D), device=device),
           "z": normal_bf16(seed, f"{name}.z", (1, hist, D), device=device)}
    if kind == 4:
        raw["ik"] = normal_bf16(seed, f"{name}.ik", (1, hist, Di), device=device)
        raw["iz"] = normal_bf16(seed, f"{name}.iz", (1, hist, Di), device=device)
    n_full = hist // r
    offs = capacity_offsets([L // r], slack=slack)
    W = shape.W
    swa = torch.zeros(1, W, D, dtype=torch.bfloat16, device=device)
    for p in range(max(0, hist - W), hist):
        swa[0, p % W] = raw["kv"][0, p]
    ring = lambda t: _ring_from_history(t, n_full * r, hist, r)
    st = LayerState(
        kind=kind, ratio=r, shape=shape,
        seq_len_in=torch.tensor([hist], dtype=torch.int32, device=device),
        pool_offsets=offs.to(device),
        swa=swa, kv_ring=ring(raw["kv"]), z_ring=ring(raw["z"]),
        kv_pool=torch.zeros(int(offs[-1]), D, dtype=torch.bfloat16, device=device),
        b_kv=normal(seed, f"{name}.b_kv", (r, D), std=0.5, device=device),
        kv_new=normal_bf16(seed, f"{name}.kv_new", (1, D), device=device),
        z_new=normal_bf16(seed, f"{name}.z_new", (1, D), device=device),
        q=normal_bf16(seed, f"{name}.q", (1, shape.Hq, D), device=device))
    if kind == 4:
        st.ik_ring, st.iz_ring = ring(raw["ik"]), ring(raw["iz"])
        st.key_pool = torch.zeros(int(offs[-1]), Di, dtype=torch.bfloat16, device=device)
        st.b_ik = normal(seed, f"{name}.b_ik", (r, Di), std=0.5, device=device)
        st.ik_new = normal_bf16(seed, f"{name}.ik_new", (1, Di), device=device)
        st.iz_new = normal_bf16(seed, f"{name}.iz_new", (1, Di), device=device)
        st.iq = normal_bf16(seed, f"{name}.iq", (1, shape.Hi, Di), device=device)
        st.w = uniform(seed, f"{name}.w", (1, shape.Hi), device=device)
    return st, raw


def _ring_from_history(t: torch.Tensor, start: int, end: int, r: int) -> torch.Tensor:
    """In-flight block ring [1, r, C]: tokens [start, end) of the history at slot pos mod r."""
    ring = torch.zeros(1, r, t.shape[2], dtype=t.dtype, device=t.device)
    for p in range(start, end):
        ring[0, p % r] = t[0, p]
    return ring


def filled_state(seed: int, kind: int, shape: LayerShape, L: torch.Tensor, device="cpu",
                 name: str = "c4layer", T: int = 1) -> LayerState:
    """A batch of sequences at context lengths L (tokens after this step, which
    appends T tokens) whose pools, rings and SWA windows are filled directly
    with N(0,1) bf16 values (the large workloads: no history is compressed).
    With T > 1 the per-token inputs get a token axis and the window ring
    W + T - 1 rows; T = 1 draws exactly what it always drew."""
    r = kind
    D, Di, W = shape.Dqk, shape.Di, shape.W
    B = L.numel()
    Lin = (L.to(torch.int64) - T)
    counts = (L.to(torch.int64) // r)
    offs = capacity_offsets(counts.tolist(), slack=1)
    cap = int(offs[-1])
    tk = (B,) if T == 1 else (B, T)          # leading axes of the per-token inputs
    sfx = "" if T == 1 else f".t{T}"
    st = LayerState(
        kind=kind, ratio=r, shape=shape,
        seq_len_in=Lin.to(torch.int32).to(device),
        pool_offsets=offs.to(device),
        swa=normal_bf16(seed, f"{name}.swa", (B, W + T - 1, D), device=device),
        kv_ring=normal_bf16(seed, f"{name}.kv_ring", (B, r, D), device=device),
        z_ring=normal_bf16(seed, f"{name}.z_ring", (B, r, D), device=device),
        kv_pool=normal_bf16(seed, f"{name}.kv_pool", (cap, D), device=device),
        b_kv=normal(seed, f"{name}.b_kv", (r, D), std=0.5, device=device),
        kv_new=normal_bf16(seed, f"{name}.kv_new{sfx}", tk + (D,), device=device),
        z_new=normal_bf16(seed, f"{name}.z_new{sfx}", tk + (D,), device=device),
        q=normal_bf16(seed, f"{name}.q{sfx}", tk + (shape.Hq, D), device=device), T=T)
    if kind == 4:
        st.ik_ring = normal_bf16(seed, f"{name}.ik_ring", (B, r, Di), device=device)
        st.iz_ring = normal_bf16(seed, f"{name}.iz_ring", (B, r, Di), device=device)
        st.key_pool = normal_bf16(seed, f"{name}.key_pool", (cap, Di), device=device)
        st.b_ik = normal(seed, f"{name}.b_ik", (r, Di), std=0.5, device=device)
        st.ik_new = normal_bf16(seed, f"{name}.ik_new{sfx}", tk + (Di,), device=device)
        st.iz_new = normal_bf16(seed, f"{name}.iz_new{sfx}", tk + (Di,), device=device)
        st.iq = normal_bf16(seed, f"{name}.iq{sfx}", tk + (shape.Hi, Di), device=device)
        st.w = uniform(seed, f"{name}.w{sfx}", tk + (shape.Hi,), device=device)
    return st
