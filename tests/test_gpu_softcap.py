"""Logit cap (softcap) on the GPU against the fp64 oracle.

attn_fwd_ex + attn_bwd_ex with softcap > 0 (through the binding's
``softcap=``): the logits s = scale q.k become c tanh(s / c), and the backward
multiplies dS by 1 - tanh^2.  The caps here are small enough (1.5 to 5) that
logits of N(0, 1) inputs reach the saturating part of tanh.
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
    # B, Hq, Hk, Sq, Sk, D, dtype, causal, window, cap, deterministic
    (1, 4, 2, 600, 600, 128, "bf16", True, None, 1.5, False),
    (2, 4, 4, 513, 700, 64, "fp16", False, None, 1.5, False),
    (1, 8, 2, 700, 700, 128, "bf16", True, (200, -1), 2.0, True),
    (1, 2, 2, 1000, 1000, 128, "bf16", False, None, 5.0, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"cap{i}" for i in range(len(CASES))])
def test_softcap_against_oracle(case):
    b, hq, hk, sq, sk, d, dt, causal, window, cap, det = case
    w = synth.small("cap", b, hq, hk, sq, sk, d, dt, causal, 400 + sum(case[:5]))
    x = synth.make_inputs(w)
    # logits of size ~2 so that tanh(s / c) saturates for the small caps
    q = (x.q.float() * 2).to(x.q.dtype)
    qd, k, v, do = (t.cuda() for t in (q, x.k, x.v, x.do))
    o, lse = ab.attn_fwd(qd, k, v, causal=causal, window=window, softcap=cap)
    runs = []
    for _ in range(2 if det else 1):
        outs = ab.attn_bwd(qd, k, v, o, lse, do, causal=causal, window=window, softcap=cap,
                           deterministic=det)
        ab.check_device_status()
        runs.append(outs)
    if det:
        for a, r in zip(*runs):
            assert torch.equal(a, r)
    ref = attn_oracle.mha_backward(q, x.k, x.v, x.do, w.scale, causal, window=window,
                                   softcap=cap)
    assert_close("softcap O", o, ref["O"])
    fin = np.isfinite(ref["LSE"])
    assert np.abs(lse.cpu().double().numpy()[fin] - ref["LSE"][fin]).max() < 1e-3
    floor = float(np.abs(ref["dV"]).max())
    for name, got in zip(("dQ", "dK", "dV"), runs[0]):
        assert_close(f"softcap {name}", got, ref[name], floor=floor)


def test_softcap_varlen():
    lens = [300, 17, 640, 129]
    w = synth.Workload("capvl", 0, 4, 2, 0, 0, 128, "bf16", True, 411, n_seqs=len(lens),
                       len_lo=1, len_hi=700)
    x = synth.make_inputs(w, lengths=lens)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    kw = dict(cu_seqlens_q=x.cu_seqlens_q.cuda(), cu_seqlens_k=x.cu_seqlens_k.cuda(),
              max_seqlen_q=max(lens), max_seqlen_k=max(lens), causal=True, softcap=1.0)
    o, lse = ab.attn_fwd(q, k, v, **kw)
    dq, dk, dv = ab.attn_bwd(q, k, v, o, lse, do, **kw)
    ab.check_device_status()
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, True, x.cu_seqlens_q,
                                   x.cu_seqlens_k, softcap=1.0)
    floor = float(np.abs(ref["dV"]).max())
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert_close(f"softcap varlen {name}", got, ref[name], floor=floor)


INSTANCES = [(dt, d, cap, left) for dt in ("bf16", "fp16") for d in (64, 128)
             for cap in (0.0, 2.0) for left in (-1, 150)] + \
    [(dt, 96, 0.0, -1) for dt in ("bf16", "fp16")]  # the D = 96 kernel: no cap, no left side


@pytest.mark.parametrize("dt,d,cap,left", INSTANCES,
                         ids=[f"{c[0]}_d{c[1]}_cap{c[2]:g}_left{c[3]}" for c in INSTANCES])
def test_every_main_kernel_instance(dt, d, cap, left):
    """The main kernel is instantiated per dtype, head dim, logit cap on/off and
    left window side present/absent (D = 96 without either): each of the eighteen
    against the oracle on a causal problem whose window edge and diagonal cut
    through tiles."""
    w = synth.small("inst", 1, 4, 2, 401, 401, d, dt, True, 500 + d + int(cap) + (left > 0))
    x = synth.make_inputs(w)
    q = (x.q.float() * 2).to(x.q.dtype) if cap else x.q
    window = (left, -1) if left >= 0 else None
    qd, k, v, do = (t.cuda() for t in (q, x.k, x.v, x.do))
    o, lse = ab.attn_fwd(qd, k, v, causal=True, window=window, softcap=cap)
    got = ab.attn_bwd(qd, k, v, o, lse, do, causal=True, window=window, softcap=cap)
    ab.check_device_status()
    ref = attn_oracle.mha_backward(q, x.k, x.v, x.do, w.scale, True, window=window, softcap=cap)
    floor = float(np.abs(ref["dV"]).max())
    for name, t in zip(("dQ", "dK", "dV"), got):
        assert_close(f"instance {name}", t, ref[name], floor=floor)
