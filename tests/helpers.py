"""Shared test helpers: bf16 bit conversions and fixture loading (no method arithmetic)."""
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def closed_form(expr: str) -> float:
    """Evaluate a closed-form expression from a golden file (exp/log/sqrt/float only)."""
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp, "log": math.log, "sqrt": math.sqrt,
                                                   "float": float}))


def as_float(v):
    return float(v) if not isinstance(v, str) else float(v.replace("inf", "inf"))


def bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of a torch bf16 tensor or of values exactly representable in bf16."""
    t = x if isinstance(x, torch.Tensor) else torch.tensor(np.asarray(x, dtype=np.float32))
    t = t.to(torch.bfloat16).contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """float64 values of bf16 bit patterns (via torch, not the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def np_state(st):
    """numpy copy of a synth.LayerState for the oracle (bf16 as uint16 bits)."""
    out = {k: (bf16_bits(v) if v.dtype == torch.bfloat16 else v.detach().cpu().numpy().copy())
           for k, v in st.tensors().items()}
    out.update(kind=st.kind, ratio=st.ratio, Dv=st.shape.Dv, k=st.shape.k, scale=st.shape.scale)
    out["key_fp8"] = getattr(st, "key_scale", None) is not None
    out["T"] = getattr(st, "T", 1)
    out["W"] = st.shape.W
    return out


def set_agreement(idx_a, idx_b, counts, k):
    """Mean over rows of |A ∩ B| / min(k, N_b) (rows with N_b = 0 count as 1)."""
    vals = []
    for b in range(idx_a.shape[0]):
        m = min(k, int(counts[b]))
        if m == 0:
            vals.append(1.0)
            continue
        a = set(int(x) for x in idx_a[b] if x >= 0)
        c = set(int(x) for x in idx_b[b] if x >= 0)
        vals.append(len(a & c) / m)
    return float(np.mean(vals))
