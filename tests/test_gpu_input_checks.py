"""Device-side checks of cu_seqlens (the packed layout's sequence offsets).

cu_seqlens live in device memory, so they are checked there: a one-block kernel
of each call checks them (start 0, nondecreasing, end = total rows, no
sequence longer than max_seqlen) before the other kernels run, and on a
violation every later kernel of the call returns at once, so the outputs keep
what they held.  attn_check_device_status reports the violation as
ATTN_ERR_ARG, names the array and clears the status; the next call runs
normally.  Every bad array below has batch + 1 entries, so the checking kernel
reads only inside it.
"""
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth

pytestmark = pytest.mark.gpu

TOTAL, MAXLEN = 300, 200
BAD_CU = {
    "first_not_zero": [4, 100, 200, 300],
    "decreasing": [0, 150, 100, 300],
    "end_not_total": [0, 100, 200, 290],
    "longer_than_max": [0, 50, 260, 300],
}


def _inputs():
    w = synth.Workload("cuchk", 0, 4, 2, 0, 0, 128, "bf16", True, 901, n_seqs=3, len_lo=100,
                       len_hi=100)
    x = synth.make_inputs(w, lengths=[100, 100, 100])
    return [t.cuda() for t in (x.q, x.k, x.v, x.do)], x.cu_seqlens_q.cuda()


@pytest.mark.parametrize("name", sorted(BAD_CU))
def test_bad_cu_seqlens_backward_is_reported(name):
    (q, k, v, do), good = _inputs()
    o = torch.randn_like(q)
    lse = torch.zeros(q.shape[1], TOTAL, device="cuda")
    bad = torch.tensor(BAD_CU[name], dtype=torch.int32, device="cuda")
    outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    ab.attn_bwd(q, k, v, o, lse, do, causal=True, cu_seqlens_q=bad, cu_seqlens_k=bad,
                max_seqlen_q=MAXLEN, max_seqlen_k=MAXLEN, dq=outs[0], dk=outs[1], dv=outs[2])
    with pytest.raises(ab.AttnError) as e:
        ab.check_device_status()
    assert e.value.code == -9 and "cu_seqlens" in str(e.value)
    for t in outs:  # no kernel after the check wrote anything
        assert t.isnan().all()
    # the status was cleared: the same call with valid offsets runs and writes every row
    o2, lse2 = ab.attn_fwd(q, k, v, causal=True, cu_seqlens_q=good, cu_seqlens_k=good,
                           max_seqlen_q=100, max_seqlen_k=100)
    ab.attn_bwd(q, k, v, o2, lse2, do, causal=True, cu_seqlens_q=good, cu_seqlens_k=good,
                max_seqlen_q=100, max_seqlen_k=100, dq=outs[0], dk=outs[1], dv=outs[2])
    ab.check_device_status()
    for t in outs:
        assert t.isfinite().all()


def test_bad_cu_seqlens_forward_is_reported():
    (q, k, v, _), _ = _inputs()
    bad = torch.tensor(BAD_CU["end_not_total"], dtype=torch.int32, device="cuda")
    o = torch.full_like(q, float("nan"))
    ab.attn_fwd(q, k, v, cu_seqlens_q=bad, cu_seqlens_k=bad, max_seqlen_q=MAXLEN,
                max_seqlen_k=MAXLEN, out=o)
    with pytest.raises(ab.AttnError) as e:
        ab.check_device_status()
    assert e.value.code == -9 and "cu_seqlens" in str(e.value)
    assert o.isnan().all()
    ab.check_device_status()
