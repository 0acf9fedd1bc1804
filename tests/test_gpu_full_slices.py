"""The full-size benchmark workloads against the fp64 oracle on whole slices.

Each test runs one workload at its full size through the calls bench.py times
(attn_fwd -> attn_bwd through the C ABI) and compares EVERY row of dQ, dK and
dV of chosen (sequence, head) slices, element by element, with the plain fp64
definition of the gradient (``attn_oracle.head_backward`` per query head,
dK and dV summed over the query heads of a key/value group).  Tolerance: the
stated rel-L2 <= 1e-2 and max-abs <= 2e-2 * max|ref| per gradient and slice.

Slices:
  * GQA B=2, Hq=32, Hk=8, S=8192, D=128, bf16, causal, deterministic off and on:
    the (sequence, kv head) groups (0, 0) and (1, 7), all four query heads each;
    deterministic mode is also compared bit for bit with a second run.
  * MHA B=2, H=16, S=4096, D=128, bf16, causal and not, and D=96 causal (its own
    kernel): heads (0, 0), (0, 9), (1, 4), (1, 15).
  * varlen, 16 packed sequences of lengths drawn from [128, 8192]: the
    shortest and the longest sequence, two heads each.
And the properties that hold at any size, on every head of the GQA workload:
sum_j dV_j = sum over the group of sum_i dO_i (rows of P sum to one), and
sum_j dK_j = 0 (rows of dS sum to zero).
"""
import functools

import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu

GQA = "gqa_b2_hq32_hk8_s8192_d128_bf16_causal"
GQA_DET = "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_det"
VARLEN = "varlen16_h16_d128_bf16_causal"


@functools.lru_cache(maxsize=2)
def _inputs(name):
    # the deterministic GQA workload draws the same tensors as the default one
    return synth.make_inputs(synth.WORKLOADS[name])


def _np(t):
    return t.double().numpy()


@functools.lru_cache(maxsize=16)
def _group_ref(name, b, g):
    """fp64 oracle gradients of every row of the (sequence b, kv head g) group of
    a padded workload: dQ [G, S, D] of its G query heads, dK and dV [S, D]
    summed over them."""
    w = synth.WORKLOADS[name]
    x = _inputs(name)
    grp = w.h_q // w.h_k
    kg, vg = _np(x.k[b, :, g]), _np(x.v[b, :, g])
    dq, dk, dv = [], 0.0, 0.0
    for h in range(g * grp, (g + 1) * grp):
        r = attn_oracle.head_backward(_np(x.q[b, :, h]), kg, vg, _np(x.do[b, :, h]), w.scale,
                                      w.causal)
        dq.append(r["dQ"])
        dk = dk + r["dK"]
        dv = dv + r["dV"]
    return np.stack(dq), dk, dv


def _run(w, x, deterministic):
    (q, k, v, do), cu_q, cu_k = to_dev(x)
    mq = mk = max(x.lengths) if w.varlen else None
    o, lse = ab.attn_fwd(q, k, v, causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                         max_seqlen_q=mq, max_seqlen_k=mk)
    outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    ab.attn_bwd(q, k, v, o, lse, do, causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                max_seqlen_q=mq, max_seqlen_k=mk, deterministic=deterministic, dq=outs[0],
                dk=outs[1], dv=outs[2])
    ab.check_device_status()
    return outs


def _compare_group(name, w, dq, dk, dv, b, g, tag):
    grp = w.h_q // w.h_k
    dq_ref, dk_ref, dv_ref = _group_ref(name, b, g)
    got_dq = dq[b, :, g * grp:(g + 1) * grp].transpose(0, 1)  # [G, S, D]
    assert_close(f"{tag} dQ b={b} g={g}", got_dq, dq_ref)
    assert_close(f"{tag} dK b={b} g={g}", dk[b, :, g], dk_ref)
    assert_close(f"{tag} dV b={b} g={g}", dv[b, :, g], dv_ref)


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
def test_gqa_s8192_whole_groups(deterministic):
    w = synth.WORKLOADS[GQA_DET if deterministic else GQA]
    x = _inputs(GQA)
    dq, dk, dv = _run(w, x, deterministic)
    for t in (dq, dk, dv):
        assert not t.isnan().any()
    for b, g in ((0, 0), (1, 7)):
        _compare_group(GQA, w, dq, dk, dv, b, g, w.name)
    if deterministic:
        again = _run(w, x, True)
        for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), again):
            assert torch.equal(a, r), f"deterministic {name} differs between runs"


@pytest.mark.parametrize("name", ["mha_b2_h16_s4096_d128_bf16",
                                  "mha_b2_h16_s4096_d128_bf16_causal",
                                  "mha_b2_h16_s4096_d96_bf16_causal"])
def test_mha_s4096_whole_heads(name):
    w = synth.WORKLOADS[name]
    x = _inputs(name)
    dq, dk, dv = _run(w, x, False)
    for b, h in ((0, 0), (0, 9), (1, 4), (1, 15)):
        _compare_group(name, w, dq, dk, dv, b, h, name)


def test_varlen_whole_sequences():
    w = synth.WORKLOADS[VARLEN]
    x = _inputs(VARLEN)
    dq, dk, dv = _run(w, x, False)
    cu = [int(c) for c in x.cu_seqlens_q]
    lens = x.lengths
    for bsel, heads in ((int(np.argmin(lens)), (3, 10)), (int(np.argmax(lens)), (0, 12))):
        lo, hi = cu[bsel], cu[bsel + 1]
        for h in heads:
            r = attn_oracle.head_backward(_np(x.q[lo:hi, h]), _np(x.k[lo:hi, h]),
                                          _np(x.v[lo:hi, h]), _np(x.do[lo:hi, h]), w.scale,
                                          w.causal)
            tag = f"varlen seq {bsel} (L={hi - lo}) head {h}"
            assert_close(f"{tag} dQ", dq[lo:hi, h], r["dQ"])
            assert_close(f"{tag} dK", dk[lo:hi, h], r["dK"])
            assert_close(f"{tag} dV", dv[lo:hi, h], r["dV"])


def test_gqa_s8192_invariants_every_head():
    """sum_j dV_j equals the group's sum_i dO_i and sum_j dK_j = 0, for every
    (sequence, kv head) of the full-size GQA workload."""
    w = synth.WORKLOADS[GQA]
    x = _inputs(GQA)
    dq, dk, dv = _run(w, x, False)
    grp = w.h_q // w.h_k
    do = x.do.cuda().double()
    sdo = do.sum(dim=1).view(w.batch, w.h_k, grp, w.head_dim).sum(dim=2)  # [B, Hk, D]
    sdv = dv.double().sum(dim=1)                                          # [B, Hk, D]
    tol = 2e-2 * sdo.abs().amax(dim=-1, keepdim=True)
    assert ((sdv - sdo).abs() <= tol).all(), (sdv - sdo).abs().max().item()
    sdk = dk.double().sum(dim=1)
    scale_k = dk.double().abs().sum(dim=1).amax(dim=-1, keepdim=True)
    assert (sdk.abs() <= 2e-2 * scale_k).all(), (sdk.abs() / scale_k).max().item()
