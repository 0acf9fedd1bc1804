"""attn_bwd_noalloc: the backward for callers that must not allocate device
memory (their memory belongs to a pool or arena owned by someone else).

It runs the same kernels as attn_bwd with the library's static 32 MiB scratch
array as workspace.  Its results are compared with attn_bwd's (which gets a
caller-provided workspace) on two calls in a row, since every call reuses
the array the previous one left behind.  This file is named to be collected
last, so a run that stops at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import binding, synth
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _entry():
    f = binding.lib().attn_bwd_noalloc
    T, P, I = binding._T, binding._P, binding._I
    f.argtypes = [T, T, T, T, P, T, T, T, T, I, I, I, I, I, I, I, ctypes.c_float, I, P, P, I, I,
                  I, P]
    f.restype = I
    return f


def _call(f, q, k, v, o, lse, do, dq, dk, dv, causal, deterministic, seqlen_q=None):
    b, sq, hq, d = q.shape
    sk, hk = k.shape[1], k.shape[2]
    sq = sq if seqlen_q is None else seqlen_q
    descs = [binding._desc(t) for t in (q, k, v, o)]
    rest = [binding._desc(t) for t in (do, dq, dk, dv)]
    return f(*(ctypes.byref(x) for x in descs), lse.data_ptr(), *(ctypes.byref(x) for x in rest),
             binding._dtype_code(q), b, sq, sk, hq, hk, d, d ** -0.5, int(causal), None, None, sq,
             sk, int(deterministic), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("deterministic,d", [(False, 128), (True, 128), (False, 192), (True, 256)],
                         ids=["d128", "d128-det", "d192", "d256-det"])
def test_noalloc_matches_attn_bwd_on_two_calls(deterministic, d):
    w = synth.small("noalloc", 2, 4, 2, 300, 300, d, "bf16", True, 123 + d)
    x = synth.make_inputs(w)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    o, lse = ab.attn_fwd(q, k, v, causal=True)
    ref = ab.attn_bwd(q, k, v, o, lse, do, causal=True, deterministic=deterministic)
    ab.check_device_status()
    f = _entry()
    for _ in range(2):
        got = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        rc = _call(f, q, k, v, o, lse, do, *got, True, deterministic)
        assert rc == 0, binding.lib().attn_last_error()
        ab.check_device_status()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(f"noalloc {name}", g, r.float().cpu().double().numpy())
            if deterministic:  # same kernels, same order of the dQ adds
                assert torch.equal(g, r), name


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_varlen_matches_attn_bwd_on_two_calls(deterministic):
    """Packed sequences (cu_seqlens) through the static scratch: ragged lengths,
    an empty sequence, and a GQA group, compared with attn_bwd's results."""
    lens = [300, 0, 129, 77]
    w = synth.Workload("noalloc_vl", 0, 4, 2, 0, 0, 128, "bf16", True, 124, n_seqs=len(lens),
                       len_lo=0, len_hi=300)
    x = synth.make_inputs(w, lengths=lens)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    cu = x.cu_seqlens_q.cuda()
    mx = max(lens)
    o, lse = ab.attn_fwd(q, k, v, causal=True, cu_seqlens_q=cu, cu_seqlens_k=cu,
                         max_seqlen_q=mx, max_seqlen_k=mx)
    ref = ab.attn_bwd(q, k, v, o, lse, do, causal=True, cu_seqlens_q=cu, cu_seqlens_k=cu,
                      max_seqlen_q=mx, max_seqlen_k=mx, deterministic=deterministic)
    ab.check_device_status()
    f = _entry()
    total, hq, d = q.shape
    hk = k.shape[1]
    for _ in range(2):
        got = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        descs = [binding._desc(t) for t in (q, k, v, o)]
        rest = [binding._desc(t) for t in (do, *got)]
        rc = f(*(ctypes.byref(t) for t in descs), lse.data_ptr(),
               *(ctypes.byref(t) for t in rest), binding._dtype_code(q), len(lens), total, total,
               hq, hk, d, d ** -0.5, 1, cu.data_ptr(), cu.data_ptr(), mx, mx, int(deterministic),
               torch.cuda.current_stream().cuda_stream)
        assert rc == 0, binding.lib().attn_last_error()
        ab.check_device_status()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(f"noalloc varlen {name}", g, r.float().cpu().double().numpy())
            if deterministic:
                assert torch.equal(g, r), name


def test_noalloc_rejects_problems_beyond_its_scratch():
    q = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 64, device="cuda")
    f = _entry()
    # claim 2^20 query rows: about 1 GiB of workspace, far beyond 32 MiB
    rc = _call(f, q, q, q, q, lse, q, q, q, q, False, False, seqlen_q=1 << 20)
    assert rc == -6
    assert b"static scratch" in binding.lib().attn_last_error()
