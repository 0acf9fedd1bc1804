"""Per-sequence used lengths (seqused_q / seqused_k) on the GPU against the oracle.

Sequence b is the first seqused[b] rows of its padded slab or packed range.
The unused rows hold other (finite) values, which must not change anything,
and the output rows past the used lengths start as NaN and must stay so (they
are not written).  A used length beyond the sequence's rows is reported by the
device-side check.
"""
import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _scramble_unused(x, used, rows_of, starts=None):
    """Unused rows of every sequence: other values, so a leak would show."""
    g = torch.Generator().manual_seed(5)
    for b, u in enumerate(used):
        r0 = 0 if starts is None else starts[b]
        n = rows_of(b)
        if u < n:
            sl = (b, slice(u, n)) if starts is None else (slice(r0 + u, r0 + n),)
            x[sl] = (torch.randn(x[sl].shape, generator=g) * 3).to(x.dtype)


@pytest.mark.parametrize("causal,det,d", [(True, False, 128), (False, False, 128), (True, True, 128),
                                         (True, False, 96), (True, False, 192), (False, True, 256)],
                         ids=["causal", "full", "causal-det", "d96", "d192", "d256-full-det"])
def test_seqused_padded(causal, det, d):
    b, hq, hk, sq, sk = 3, 8, 2, 700, 700
    uq, uk = [650, 0, 700], [600, 300, 129]
    w = synth.small("used", b, hq, hk, sq, sk, d, "bf16", causal, 611 + d)
    x = synth.make_inputs(w)
    for t, u in ((x.q, uq), (x.do, uq), (x.k, uk), (x.v, uk)):
        _scramble_unused(t, u, lambda _: t.shape[1])
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    used_q = torch.tensor(uq, dtype=torch.int32, device="cuda")
    used_k = torch.tensor(uk, dtype=torch.int32, device="cuda")
    o = torch.full_like(q, float("nan"))
    lse = torch.full((b, hq, sq), float("nan"), device="cuda")
    ab.attn_fwd(q, k, v, causal=causal, out=o, lse=lse, seqused_q=used_q, seqused_k=used_k)
    runs = []
    for _ in range(2 if det else 1):
        outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        ab.attn_bwd(q, k, v, o, lse, do, causal=causal, deterministic=det, dq=outs[0],
                    dk=outs[1], dv=outs[2], seqused_q=used_q, seqused_k=used_k)
        ab.check_device_status()
        runs.append(outs)
    if det:
        for a, r in zip(*runs):
            assert torch.equal(a.nan_to_num(7.0), r.nan_to_num(7.0))
    dq, dk, dv = runs[0]
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, causal, seqused_q=uq,
                                   seqused_k=uk)
    floor = float(np.abs(ref["dV"]).max())
    for bb in range(b):
        for t in (dq, o):
            assert t[bb, uq[bb]:].isnan().all() and not t[bb, :uq[bb]].isnan().any()
        for t in (dk, dv):
            assert t[bb, uk[bb]:].isnan().all() and not t[bb, :uk[bb]].isnan().any()
        if uq[bb]:
            assert_close(f"used O {bb}", o[bb, :uq[bb]], ref["O"][bb, :uq[bb]])
            assert_close(f"used dQ {bb}", dq[bb, :uq[bb]], ref["dQ"][bb, :uq[bb]], floor=floor)
        if uk[bb]:
            assert_close(f"used dK {bb}", dk[bb, :uk[bb]], ref["dK"][bb, :uk[bb]], floor=floor)
            assert_close(f"used dV {bb}", dv[bb, :uk[bb]], ref["dV"][bb, :uk[bb]], floor=floor)


def test_seqused_varlen():
    cq = [0, 300, 600, 1000]
    uq, uk = [250, 0, 400], [300, 120, 64]
    lens = [cq[i + 1] - cq[i] for i in range(3)]
    w = synth.Workload("usedvl", 0, 4, 2, 0, 0, 128, "bf16", True, 612, n_seqs=3, len_lo=0,
                       len_hi=400)
    x = synth.make_inputs(w, lengths=lens)
    for t, u in ((x.q, uq), (x.do, uq), (x.k, uk), (x.v, uk)):
        _scramble_unused(t, u, lambda bb: lens[bb], starts=cq)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    kw = dict(cu_seqlens_q=x.cu_seqlens_q.cuda(), cu_seqlens_k=x.cu_seqlens_k.cuda(),
              max_seqlen_q=max(lens), max_seqlen_k=max(lens), causal=True,
              seqused_q=torch.tensor(uq, dtype=torch.int32, device="cuda"),
              seqused_k=torch.tensor(uk, dtype=torch.int32, device="cuda"))
    o, lse = ab.attn_fwd(q, k, v, **kw)
    outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    ab.attn_bwd(q, k, v, o, lse, do, dq=outs[0], dk=outs[1], dv=outs[2], **kw)
    ab.check_device_status()
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, True, x.cu_seqlens_q,
                                   x.cu_seqlens_k, seqused_q=uq, seqused_k=uk)
    floor = float(np.abs(ref["dV"]).max())
    for bb in range(3):
        qs, ks = slice(cq[bb], cq[bb] + uq[bb]), slice(cq[bb], cq[bb] + uk[bb])
        assert outs[0][cq[bb] + uq[bb]:cq[bb + 1]].isnan().all()
        assert outs[1][cq[bb] + uk[bb]:cq[bb + 1]].isnan().all()
        for name, got, key, sl in (("dQ", outs[0], "dQ", qs), ("dK", outs[1], "dK", ks),
                                   ("dV", outs[2], "dV", ks)):
            if sl.stop > sl.start:
                assert_close(f"used varlen {name} {bb}", got[sl], ref[key][sl], floor=floor)


def test_seqused_beyond_rows_is_reported():
    q = torch.randn(2, 128, 2, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = ab.attn_fwd(q, q, q)
    bad = torch.tensor([128, 129], dtype=torch.int32, device="cuda")
    ab.attn_bwd(q, q, q, o, lse, q, seqused_q=bad)
    with pytest.raises(ab.AttnError) as e:
        ab.check_device_status()
    assert e.value.code == -9 and "seqused_q" in str(e.value)
    ab.check_device_status()  # the status was cleared by the report
