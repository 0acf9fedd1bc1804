"""Head dimensions above 128 (up to 256, multiples of 8) against the fp64 oracle.

The CK wrapper's argument checks (flash-attention csrc/flash_attn_ck/mha_bwd.cpp,
mha_bwd) accept head_size % 8 == 0 and head_size <= 256, and the FA3 launcher
(hopper/flash_bwd_launch_template.h) dispatches backward kernels for 192 and
256.  Here the backward for D in (128, 256] runs in two passes (dV and dK/dQ)
on tiles of 64-column chunks: three chunks for D <= 192, four above, with the
columns past D zero; the forward streams K and V in 64-column chunks.
Tolerance as everywhere: rel-L2 <= 1e-2, max-abs <= 2e-2 * max|ref| per
gradient; O and LSE as in the forward test.
"""
import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu


def _run(w, x, deterministic=False, window=None, softcap=0.0, secondary=False):
    (q, k, v, do), cu_q, cu_k = to_dev(x)
    mq = max(x.lengths) if cu_q is not None else None
    mk = max(x.lengths_k) if cu_q is not None else None
    kw = dict(causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=mq,
              max_seqlen_k=mk, window=window, softcap=softcap)
    if secondary:  # the oracle's O (rounded) and LSE: isolates the backward
        o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, w.causal, x.cu_seqlens_q,
                                                 x.cu_seqlens_k, window=window, softcap=softcap)
        o = torch.tensor(o_ref).to(q.dtype).cuda()
        lse = torch.tensor(lse_ref, dtype=torch.float32).cuda()
    else:
        o, lse = ab.attn_fwd(q, k, v, **kw)
    outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    ab.attn_bwd(q, k, v, o, lse, do, deterministic=deterministic, dq=outs[0], dk=outs[1],
                dv=outs[2], **kw)
    ab.check_device_status()
    return outs, o, lse


def _check(w, x, outs, window=None, softcap=0.0, tag=""):
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, w.causal, x.cu_seqlens_q,
                                   x.cu_seqlens_k, window=window, softcap=softcap)
    floor = float(np.abs(ref["dV"]).max())
    for name, got in zip(("dQ", "dK", "dV"), outs):
        assert not got.isnan().any(), f"{tag} {name}: unwritten rows"
        assert_close(f"{tag} {name}", got, ref[name], floor=floor)
    return ref


CASES = [
    # B, Hq, Hk, Sq, Sk, D, dtype, causal
    (1, 2, 2, 128, 128, 256, "bf16", False),
    (2, 4, 2, 300, 300, 256, "bf16", True),     # GQA, ragged last tile
    (1, 2, 2, 65, 65, 256, "fp16", True),
    (1, 8, 2, 520, 520, 256, "bf16", True),     # GQA 4:1, several tiles
    (1, 2, 1, 1, 1, 256, "bf16", False),
    (1, 2, 2, 100, 300, 256, "bf16", True),     # Sq < Sk, bottom-right causal
    (1, 2, 2, 300, 100, 256, "fp16", True),     # Sq > Sk: leading rows see no key
    (1, 4, 2, 384, 384, 192, "bf16", True),     # D = 192: three chunks, none padded
    (2, 2, 2, 257, 257, 192, "fp16", False),
    (1, 4, 2, 300, 100, 192, "bf16", True),     # Sq > Sk at three chunks
    (1, 8, 2, 520, 520, 160, "bf16", True),     # three chunks, the last half zero
    (1, 2, 2, 200, 200, 200, "fp16", False),    # just above 192: four chunks
    (1, 2, 2, 200, 200, 136, "bf16", True),     # just above 128
    (1, 2, 1, 333, 333, 248, "bf16", False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[5]}-{i}" for i, c in enumerate(CASES)])
def test_wide_head_dim_matches_oracle(case):
    b, hq, hk, sq, sk, d, dt, causal = case
    w = synth.small("wide", b, hq, hk, sq, sk, d, dt, causal, 700 + sq + sk + d)
    x = synth.make_inputs(w)
    outs, o, lse = _run(w, x)
    ref = _check(w, x, outs, tag=str(case))
    assert_close(f"{case} O", o, ref["O"])
    lc, lr = lse.cpu().double().numpy(), ref["LSE"]
    fin = np.isfinite(lr)
    assert (np.isinf(lc) == ~fin).all()
    np.testing.assert_allclose(lc[fin], lr[fin], rtol=0, atol=2e-3)


@pytest.mark.parametrize("d", [256, 192])
def test_wide_backward_alone(d):
    """The oracle's O and LSE into the GPU backward: the backward's own error."""
    w = synth.small("wide2", 1, 4, 2, 700, 700, d, "bf16", True, 811 + d)
    x = synth.make_inputs(w)
    outs, _, _ = _run(w, x, secondary=True)
    _check(w, x, outs, tag=f"secondary d={d}")


@pytest.mark.parametrize("d", [256, 192])
def test_wide_deterministic_bitwise(d):
    w = synth.small("wide_det", 1, 8, 2, 1000, 1000, d, "bf16", True, 821 + d,
                    deterministic=True)
    x = synth.make_inputs(w)
    runs = [_run(w, x, deterministic=True)[0] for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    _check(w, x, runs[0], tag="det")


@pytest.mark.parametrize("d", [256, 192])
def test_wide_varlen_cross_attention(d):
    lq, lk = [300, 0, 17, 129, 640], [200, 150, 0, 513, 64]
    w = synth.Workload("wide_vl", 0, 4, 2, 0, 0, d, "bf16", True, 831 + d, n_seqs=len(lq),
                       len_lo=0, len_hi=700)
    x = synth.make_inputs(w, lengths=lq, lengths_k=lk)
    outs, _, _ = _run(w, x)
    _check(w, x, outs, tag="varlen cross")


@pytest.mark.parametrize("window,cap,d", [((200, -1), 0.0, 256), (None, 4.0, 256),
                                         ((64, 64), 3.0, 256), ((64, 64), 3.0, 176)],
                         ids=["window", "softcap", "band+cap", "band+cap-d176"])
def test_wide_window_and_softcap(window, cap, d):
    causal = window is None or window[1] < 0
    w = synth.small("wide_wc", 1, 4, 2, 600, 600, d, "bf16", causal, 841 + d)
    x = synth.make_inputs(w)
    outs, _, _ = _run(w, x, window=window, softcap=cap)
    _check(w, x, outs, window=window, softcap=cap, tag=f"window={window} cap={cap}")


@pytest.mark.parametrize("d", [256, 192])
def test_wide_full_size_whole_heads(d):
    """MHA B=2, H=16, S=4096, D=256 and 192, bf16, causal at full size: every row
    of two whole heads against the fp64 oracle, and sum_j dV_j = sum_i dO_i on
    every head."""
    w = synth.WORKLOADS[f"mha_b2_h16_s4096_d{d}_bf16_causal"]
    x = synth.make_inputs(w)
    (dq, dk, dv), _, _ = _run(w, x)
    for b, h in ((0, 3), (1, 15)):
        r = attn_oracle.head_backward(x.q[b, :, h].double().numpy(), x.k[b, :, h].double().numpy(),
                                      x.v[b, :, h].double().numpy(), x.do[b, :, h].double().numpy(),
                                      w.scale, w.causal)
        for name, got in (("dQ", dq[b, :, h]), ("dK", dk[b, :, h]), ("dV", dv[b, :, h])):
            assert_close(f"d{d} full {name} b={b} h={h}", got, r[name])
    sdv = dv.double().sum(dim=1)
    sdo = x.do.cuda().double().sum(dim=1)
    assert ((sdv - sdo).abs() <= 2e-2 * sdo.abs().amax(dim=-1, keepdim=True)).all()
