"""fp64 CPU oracle for the fused attention backward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code with
the CUDA path; its inputs come from ``attention_backward_bwd_gb300.synth``
(random numbers only).

What it computes is the plain definition of softmax attention and of its
gradient, written out step by step in float64 with a library matmul as the
only primitive.  No tiling, no online softmax, no recomputation tricks.

Sources (page title, section):
  * test_tilelang_kernel_mha_bwd.py (TileLang), ``ref_program``: scores =
    Q K^T / sqrt(D), lower-triangular causal mask filled with -inf, softmax
    over keys, output = P V; gradients by differentiation.
  * same page, ``flashattn_bwd``: the backward steps P = softmax(S),
    dV = P^T dO, dP = dO V^T, dS = P * (dP - Delta), dK = dS^T Q, dQ = dS K,
    all times the softmax scale; ``flashattn_bwd_preprocess``: Delta =
    rowsum(O * dO).
  * flash-attention csrc/flash_attn_ck/mha_bwd.cpp, ``mha_bwd``: query head h
    reads key/value head h // (H / H_k), and dK, dV are summed over the
    H / H_k query heads of a group (the ``sum_out`` over the group dim);
    causal is a window (left, 0) in bottom-right alignment; seqlen_q == 0
    gives zero dK, dV.
  * flash-attention hopper/flash_bwd_launch_template.h, ``run_flash_bwd``:
    varlen tensors are packed [total, H, D] with per-sequence offsets from
    cu_seqlens; LSE is natural-log (the preprocess makes the log2 copy).

  * same CK page, the mask set-up of ``mha_bwd``: a local (sliding-window)
    mask is a window (left, right) around each query's aligned key, -1 meaning
    unbounded on that side, in the same bottom-right alignment; causal is the
    window (-1, 0).

  * flash-attention hopper/flash_bwd_launch_template.h: ``Has_softcap`` /
    ``params.softcap`` select a logit cap (no formula is given there);
    ``seqused_q`` / ``seqused_k`` give each sequence a used length inside its
    padded or packed rows.

Readings where the pages leave a point open:
  * causal with Sq != Sk: key j is allowed for query i iff j <= i + (Sk - Sq).
  * window (left, right): with off = Sk - Sq, key j is allowed for query i iff
    j >= i + off - left (when left >= 0) and j <= i + off + right (when
    right >= 0); causal together with a window keeps the window's left side
    and bounds the right side at 0.
  * seqused: sequence b is the first seqused[b] rows of its rows (padded slab or
    packed range); the rest of its rows take no part, and their gradients are
    left as they were (zero here).
  * softcap c > 0: the logits s = scale * q.k are capped as c * tanh(s / c)
    before the softmax (the usual logit cap); the backward multiplies dS by
    the cap's derivative 1 - tanh(s / c)^2.  c = 0 means no cap.
  * a query row with no allowed key: O = 0, LSE = +inf, dQ = 0, and it adds
    nothing to dK or dV.
  * scale defaults to 1/sqrt(D).

Every function here is pinned by ``tests/test_oracle_pins.py`` (finite
differences, algebraic identities, closed forms, an independent fp64 torch
autograd run and planted-mistake checks); ``group_backward_rows`` is pinned to
``mha_backward`` row by row.
"""
from __future__ import annotations

import numpy as np


def _window_sides(causal: bool, window) -> tuple:
    """(left, right) of the mask, -1 = unbounded; causal bounds the right at 0."""
    left, right = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    if causal:
        right = 0
    return left, right


def allowed_pairs(i, j, sq: int, sk: int, causal: bool, window=None) -> np.ndarray:
    """True where query i may attend key j (i, j broadcastable index arrays)."""
    left, right = _window_sides(causal, window)
    ok = np.ones(np.broadcast_shapes(np.shape(i), np.shape(j)), dtype=bool)
    if right >= 0:
        ok &= j <= i + (sk - sq) + right
    if left >= 0:
        ok &= j >= i + (sk - sq) - left
    return ok


def allowed_mask(sq: int, sk: int, causal: bool, window=None) -> np.ndarray:
    """Boolean [sq, sk]: True where query i may attend key j."""
    return allowed_pairs(np.arange(sq)[:, None], np.arange(sk)[None, :], sq, sk, causal, window)


def head_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool,
                 window=None, softcap: float = 0.0):
    """Forward of one head.  q [Sq, D], k and v [Sk, D], float64.

    Returns (O [Sq, D], LSE [Sq] natural log, P [Sq, Sk]).
    """
    sq, sk = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    allowed = allowed_mask(sq, sk, causal, window)
    s = np.where(allowed, s, -np.inf)
    any_key = allowed.any(axis=1) if sk > 0 else np.zeros(sq, dtype=bool)
    m = np.where(any_key, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(allowed, np.exp(s - m[:, None]), 0.0)
    ell = e.sum(axis=1)
    lse = np.where(any_key, m + np.log(np.where(any_key, ell, 1.0)), np.inf)
    p = np.where(allowed, np.exp(s - np.where(any_key, lse, 0.0)[:, None]), 0.0)
    o = p @ v
    return o, lse, p


def head_backward(q, k, v, do, scale: float, causal: bool, window=None, softcap: float = 0.0):
    """Gradient of one head, by the definition.  All arrays float64.

    Returns a dict with O, LSE, P, dP, Delta (= rowsum(P * dP)), dS, dQ, dK, dV;
    dS is the gradient with respect to the (uncapped) logits scale * q.k.
    """
    o, lse, p = head_forward(q, k, v, scale, causal, window, softcap)
    dv = p.T @ do
    dp = do @ v.T
    delta = (p * dp).sum(axis=1)
    ds = p * (dp - delta[:, None])
    if softcap > 0:
        ds = ds * (1.0 - np.tanh(scale * (q @ k.T) / softcap) ** 2)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return {"O": o, "LSE": lse, "P": p, "dP": dp, "Delta": delta, "dS": ds,
            "dQ": dq, "dK": dk, "dV": dv}


def delta_from_output(o: np.ndarray, do: np.ndarray) -> np.ndarray:
    """Delta_i = sum_d O_id * dO_id (the backward preprocess), over the last axis."""
    return (np.asarray(o, dtype=np.float64) * np.asarray(do, dtype=np.float64)).sum(axis=-1)


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _sequences(q, k, cu_q, cu_k, used_q=None, used_k=None):
    """Yield (b, q_rows, k_rows) slices for padded [B,S,H,D] or packed [total,H,D];
    ``used_q`` / ``used_k`` (per sequence) keep only each sequence's first rows."""
    uq = None if used_q is None else [int(x) for x in _f64(used_q)]
    uk = None if used_k is None else [int(x) for x in _f64(used_k)]
    if cu_q is None:
        for b in range(q.shape[0]):
            qs = slice(None) if uq is None else slice(0, uq[b])
            ks = slice(None) if uk is None else slice(0, uk[b])
            yield b, (b, qs), (b, ks)
    else:
        cq = [int(x) for x in _f64(cu_q)]
        ck = [int(x) for x in _f64(cu_k)]
        for b in range(len(cq) - 1):
            nq = cq[b + 1] - cq[b] if uq is None else uq[b]
            nk = ck[b + 1] - ck[b] if uk is None else uk[b]
            yield b, (slice(cq[b], cq[b] + nq),), (slice(ck[b], ck[b] + nk),)


def _take(x, sel, h):
    if len(sel) == 2:
        return x[sel[0], sel[1], h, :]
    return x[sel[0], h, :]


def _put(x, sel, h, val, add=False):
    if len(sel) == 2:
        if add:
            x[sel[0], sel[1], h, :] += val
        else:
            x[sel[0], sel[1], h, :] = val
    else:
        if add:
            x[sel[0], h, :] += val
        else:
            x[sel[0], h, :] = val


def mha_forward(q, k, v, scale=None, causal=False, cu_seqlens_q=None, cu_seqlens_k=None,
                heads=None, window=None, softcap=0.0, seqused_q=None, seqused_k=None):
    """Multi-head forward.  q [B,Sq,H,D] (or packed [total,H,D]), k/v with H_k heads.

    Returns (O like q, LSE [B,H,Sq] or [H,total_q]).  ``heads`` restricts the
    query heads computed (others are left zero).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    hq, hk, d = q.shape[-2], k.shape[-2], q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    g = hq // hk
    o = np.zeros_like(q)
    if cu_seqlens_q is None:
        lse = np.zeros((q.shape[0], hq, q.shape[1]))
    else:
        lse = np.zeros((hq, q.shape[0]))
    hs = range(hq) if heads is None else heads
    for b, qs, ks in _sequences(q, k, cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k):
        for h in hs:
            oh, lh, _ = head_forward(_take(q, qs, h), _take(k, ks, h // g), _take(v, ks, h // g),
                                     scale, causal, window, softcap)
            _put(o, qs, h, oh)
            if cu_seqlens_q is None:
                lse[b, h, qs[1]] = lh
            else:
                lse[h, qs[0]] = lh
    return o, lse


def mha_backward(q, k, v, do, scale=None, causal=False, cu_seqlens_q=None, cu_seqlens_k=None,
                 kv_heads=None, window=None, softcap=0.0, seqused_q=None, seqused_k=None):
    """Multi-head backward by the definition, with GQA group sums.

    Returns dict(dQ, dK, dV, O, LSE, Delta) in the input layouts (LSE/Delta as
    [B,H,Sq] or [H,total_q]).  ``kv_heads`` restricts the computation to the
    query heads of those key/value heads (others stay zero).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    hq, hk, d = q.shape[-2], k.shape[-2], q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    g = hq // hk
    dq, dk, dv, o = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(q)
    if cu_seqlens_q is None:
        lse = np.zeros((q.shape[0], hq, q.shape[1]))
    else:
        lse = np.zeros((hq, q.shape[0]))
    delta = np.zeros_like(lse)
    kvs = range(hk) if kv_heads is None else kv_heads
    for b, qs, ks in _sequences(q, k, cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k):
        for hkv in kvs:
            for h in range(hkv * g, hkv * g + g):
                r = head_backward(_take(q, qs, h), _take(k, ks, hkv), _take(v, ks, hkv),
                                  _take(do, qs, h), scale, causal, window, softcap)
                _put(dq, qs, h, r["dQ"])
                _put(o, qs, h, r["O"])
                _put(dk, ks, hkv, r["dK"], add=True)
                _put(dv, ks, hkv, r["dV"], add=True)
                if cu_seqlens_q is None:
                    lse[b, h, qs[1]] = r["LSE"]
                    delta[b, h, qs[1]] = r["Delta"]
                else:
                    lse[h, qs[0]] = r["LSE"]
                    delta[h, qs[0]] = r["Delta"]
    return {"dQ": dq, "dK": dk, "dV": dv, "O": o, "LSE": lse, "Delta": delta}


def group_backward_rows(q, k, v, do, b: int, g: int, q_rows, k_rows, scale=None,
                        causal=False, block: int = 512, window=None, softcap: float = 0.0):
    """Exact gradients at selected rows of one (sequence, kv head) group, for
    problems too large for ``mha_backward`` (padded [B,S,H,D] inputs only).

    Returns (dq_rows [G, len(q_rows), D] for the G query heads of kv head g,
    dk_rows [len(k_rows), D], dv_rows [len(k_rows), D]), float64.  The same
    definition as ``head_backward`` (softmax over all allowed keys of a query
    row, Delta = rowsum(P * dP), dS = P (dP - Delta)), evaluated for query rows
    ``block`` at a time; the blocks only bound memory, and dK, dV at the chosen
    key rows accumulate the blocks' sums over query rows in float64.
    """
    hq, hk, d = q.shape[2], k.shape[2], q.shape[3]
    scale = d ** -0.5 if scale is None else scale
    grp = hq // hk
    q_rows = [int(i) for i in q_rows]
    k_rows = np.asarray([int(j) for j in k_rows], dtype=np.int64)
    kg = _f64(k[b, :, g, :])
    vg = _f64(v[b, :, g, :])
    sq, sk = q.shape[1], kg.shape[0]
    dq = np.zeros((grp, len(q_rows), d))
    dk = np.zeros((len(k_rows), d))
    dv = np.zeros((len(k_rows), d))
    for hh in range(grp):
        h = g * grp + hh
        qh = _f64(q[b, :, h, :])
        doh = _f64(do[b, :, h, :])
        for i0 in range(0, sq, block):
            i1 = min(sq, i0 + block)
            ii = np.arange(i0, i1)[:, None]
            jj = np.arange(sk)[None, :]
            allowed = allowed_pairs(ii, jj, sq, sk, causal, window)
            s_raw = scale * (qh[i0:i1] @ kg.T)
            s = softcap * np.tanh(s_raw / softcap) if softcap > 0 else s_raw
            s = np.where(allowed, s, -np.inf)
            any_key = allowed.any(axis=1)
            m = np.where(any_key, s.max(axis=1), 0.0)
            ell = np.where(allowed, np.exp(s - m[:, None]), 0.0).sum(axis=1)
            lse = np.where(any_key, m + np.log(np.where(any_key, ell, 1.0)), 0.0)
            p = np.where(allowed, np.exp(s - lse[:, None]), 0.0)
            dp = doh[i0:i1] @ vg.T
            delta = (p * dp).sum(axis=1)
            ds = p * (dp - delta[:, None])
            if softcap > 0:
                ds = ds * (1.0 - np.tanh(s_raw / softcap) ** 2)
            for n, i in enumerate(q_rows):
                if i0 <= i < i1:
                    dq[hh, n] = scale * (ds[i - i0] @ kg)
            dk += scale * (ds[:, k_rows].T @ qh[i0:i1])
            dv += p[:, k_rows].T @ doh[i0:i1]
    return dq, dk, dv

