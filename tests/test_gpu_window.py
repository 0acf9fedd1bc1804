"""Local (sliding-window) masks on the GPU against the fp64 oracle.

attn_fwd_ex + attn_bwd_ex (through the binding's ``window=``) on shapes
that put the window's edges inside tiles, leave whole key tiles unseen
(dK = dV = 0 there) or whole query rows without keys (dQ = 0, O = 0), and in
deterministic mode, where the dQ adds of a query tile are ordered over the key
tiles inside its window.
"""
import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hk, Sq, Sk, D, dtype, causal, window, deterministic
    (1, 4, 2, 700, 700, 128, "bf16", True, (256, -1), False),    # sliding-window causal
    (2, 4, 4, 513, 513, 64, "fp16", False, (100, 37), False),    # two-sided band
    (1, 8, 2, 300, 900, 128, "bf16", False, (50, 50), False),    # Sq < Sk: early key tiles unseen
    (1, 2, 2, 900, 300, 128, "bf16", True, (17, -1), False),     # Sq > Sk: rows without keys
    (2, 4, 2, 1000, 1000, 128, "bf16", False, (0, 0), False),    # one key per query
    (1, 8, 2, 1000, 1000, 128, "bf16", True, (300, -1), True),   # deterministic, left window
    (1, 4, 4, 640, 640, 64, "bf16", False, (129, 0), True),      # deterministic, D = 64
]


def _run(x, w, window, det, o=None, lse=None):
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    kw = {}
    if x.cu_seqlens_q is not None:
        kw = dict(cu_seqlens_q=x.cu_seqlens_q.cuda(), cu_seqlens_k=x.cu_seqlens_k.cuda(),
                  max_seqlen_q=max(x.lengths), max_seqlen_k=max(x.lengths_k))
    if o is None:
        o, lse = ab.attn_fwd(q, k, v, causal=w.causal, window=window, **kw)
    outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    ab.attn_bwd(q, k, v, o, lse, do, causal=w.causal, deterministic=det, window=window,
                dq=outs[0], dk=outs[1], dv=outs[2], **kw)
    ab.check_device_status()
    return o, lse, outs


@pytest.mark.parametrize("case", CASES, ids=[f"win{i}" for i in range(len(CASES))])
def test_window_against_oracle(case):
    b, hq, hk, sq, sk, d, dt, causal, window, det = case
    w = synth.small("win", b, hq, hk, sq, sk, d, dt, causal, 200 + sum(case[:5]))
    x = synth.make_inputs(w)
    o, lse, (dq, dk, dv) = _run(x, w, window, det)
    if det:
        _, _, again = _run(x, w, window, det, o, lse)
        for a, r in zip((dq, dk, dv), again):
            assert torch.equal(a, r)
    for t in (dq, dk, dv):
        assert not t.isnan().any()
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, causal, window=window)
    assert_close("window O", o, ref["O"])
    lse_g = lse.cpu().double().numpy()
    fin = np.isfinite(ref["LSE"])
    assert (np.isinf(lse_g) == ~fin).all()
    assert np.abs(lse_g[fin] - ref["LSE"][fin]).max() < 1e-3
    floor = float(np.abs(ref["dV"]).max())
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert_close(f"window {name}", got, ref[name], floor=floor)
    # keys that no query sees, and queries that see no key, are exact zeros
    seen = attn_oracle.allowed_mask(sq, sk, causal, window)
    unseen_k = torch.from_numpy(~seen.any(axis=0)).cuda()
    keyless_q = torch.from_numpy(~seen.any(axis=1)).cuda()
    assert (dk[:, unseen_k] == 0).all() and (dv[:, unseen_k] == 0).all()
    assert (dq[:, keyless_q] == 0).all()


def test_window_cross_attention_varlen():
    lq, lk = [300, 0, 17, 640, 5], [200, 150, 40, 513, 0]
    w = synth.Workload("winvl", 0, 4, 2, 0, 0, 128, "bf16", False, 301, n_seqs=len(lq),
                       len_lo=0, len_hi=700)
    x = synth.make_inputs(w, lengths=lq, lengths_k=lk)
    _, _, (dq, dk, dv) = _run(x, w, (64, 16), False)
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, False, x.cu_seqlens_q,
                                   x.cu_seqlens_k, window=(64, 16))
    floor = float(np.abs(ref["dV"]).max())
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert_close(f"window varlen {name}", got, ref[name], floor=floor)


def test_window_wider_than_problem_equals_no_window():
    """A window that excludes nothing runs the unmasked schedule: in
    deterministic mode the results equal attn_bwd's bit for bit."""
    w = synth.small("winwide", 1, 4, 2, 500, 500, 128, "bf16", True, 77)
    x = synth.make_inputs(w)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    o, lse = ab.attn_fwd(q, k, v, causal=True)
    o2, lse2 = ab.attn_fwd(q, k, v, causal=True, window=(100000, 100000))
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    plain = ab.attn_bwd(q, k, v, o, lse, do, causal=True, deterministic=True)
    wide = ab.attn_bwd(q, k, v, o, lse, do, causal=True, deterministic=True,
                       window=(100000, -1))
    ab.check_device_status()
    for a, r in zip(plain, wide):
        assert torch.equal(a, r)
