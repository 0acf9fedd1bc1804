"""Shared helpers for the GPU parity tests (oracle comparison, tolerances)."""
from __future__ import annotations

import numpy as np
import torch

from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle

# Tolerance for fp16/bf16 gradients against the fp64 oracle: relative L2 error
# <= 1e-2 and max abs error <= 2e-2 * max|ref|, per gradient tensor.
REL_L2 = 1e-2
MAX_ABS_FRAC = 2e-2


def errors(got, ref):
    g = got.detach().float().cpu().double().numpy() if hasattr(got, "detach") else np.asarray(got)
    r = np.asarray(ref, dtype=np.float64)
    den = max(np.linalg.norm(r), 1e-30)
    rel = float(np.linalg.norm(g - r) / den)
    mx = float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-30)) if r.size else 0.0
    return rel, mx


def assert_close(name, got, ref, rel_l2=REL_L2, max_frac=MAX_ABS_FRAC, floor=None):
    """``floor``: a magnitude scale for gradients whose exact value is zero
    (e.g. dQ = dK = 0 when a row sees a single key); then only
    max|got| <= max_frac * floor is required, a relative error being undefined."""
    r = np.asarray(ref, dtype=np.float64)
    if floor is not None and r.size and np.abs(r).max() <= 1e-6 * floor:
        g = got.detach().float().cpu().double().numpy()
        assert np.abs(g).max() <= max_frac * floor, f"{name}: {np.abs(g).max():.3e} on a zero ref"
        return 0.0, float(np.abs(g).max() / floor)
    rel, mx = errors(got, ref)
    assert np.isfinite(rel) and rel <= rel_l2, f"{name}: rel-L2 {rel:.3e} > {rel_l2}"
    assert mx <= max_frac, f"{name}: max-abs/max|ref| {mx:.3e} > {max_frac}"
    return rel, mx


def to_dev(x: synth.Inputs, dev="cuda"):
    out = [t.to(dev) for t in (x.q, x.k, x.v, x.do)]
    cu_q = x.cu_seqlens_q.to(dev) if x.cu_seqlens_q is not None else None
    cu_k = x.cu_seqlens_k.to(dev) if x.cu_seqlens_k is not None else None
    return out, cu_q, cu_k


def max_len(x: synth.Inputs):
    if x.lengths is None:
        return None
    return max(x.lengths) if x.lengths else 0
