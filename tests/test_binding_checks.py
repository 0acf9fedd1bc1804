"""The binding's own argument checks (no GPU needed).

The C library receives raw pointers, so it cannot see where a tensor lives, its
dtype or its size; the binding checks those before any call, because a host
pointer handed to a kernel, or a tensor smaller than its arguments imply, would
be read or written past its end on the device.  Host tensors are the valid side
of the host-buffer entry points, so their checks run here on CPU tensors; the
device entry points are given CPU (and meta) tensors, which they must refuse.
"""
import pytest
import torch

import attention_backward_bwd_gb300 as ab

B, S, HQ, HK, D = 2, 64, 4, 2, 64


def _host(dtype=torch.bfloat16):
    q = torch.randn(B, S, HQ, D).to(dtype)
    k = torch.randn(B, S, HK, D).to(dtype)
    v = torch.randn(B, S, HK, D).to(dtype)
    o = torch.randn(B, S, HQ, D).to(dtype)
    do = torch.randn(B, S, HQ, D).to(dtype)
    lse = torch.zeros(B, HQ, S)
    return [q, k, v, o, lse, do]


def _code(fn, *a, **kw):
    with pytest.raises(ab.AttnError) as e:
        fn(*a, **kw)
    return e.value.code, str(e.value)


def test_device_entry_points_refuse_host_tensors():
    q, k, v, o, lse, do = _host()
    code, msg = _code(ab.attn_bwd, q, k, v, o, lse, do)
    assert code == -9 and "CUDA" in msg
    code, msg = _code(ab.attn_fwd, q, k, v)
    assert code == -9 and "CUDA" in msg
    m = [t.to("meta") for t in (q, k, v)]
    assert _code(ab.attn_fwd, *m)[0] == -9


def test_host_entry_points_check_dtype_shape_stride_and_lse():
    t = _host()
    # k in another dtype than q
    bad = list(t)
    bad[1] = bad[1].to(torch.float16)
    code, msg = _code(ab.attn_bwd_host, *bad)
    assert code == -1 and "k has dtype" in msg
    # dO with one position fewer than q
    bad = list(t)
    bad[5] = bad[5][:, :-1]
    code, msg = _code(ab.attn_bwd_host, *bad)
    assert code == -2 and "do has shape" in msg
    # v unlike k
    bad = list(t)
    bad[2] = torch.randn(B, S, HK, D + 8).to(torch.bfloat16)
    assert _code(ab.attn_bwd_host, *bad)[0] == -2
    # head dimension not of unit stride
    bad = list(t)
    bad[0] = torch.randn(B, S, HQ, 2 * D).to(torch.bfloat16)[..., ::2]
    code, msg = _code(ab.attn_bwd_host, *bad)
    assert code == -3 and "unit stride" in msg
    # LSE: wrong shape, wrong dtype, not contiguous
    for lse in (torch.zeros(B, S, HQ), torch.zeros(B, HQ, S, dtype=torch.float64),
                torch.zeros(B, S, HQ).transpose(1, 2)):
        bad = list(t)
        bad[4] = lse
        code, msg = _code(ab.attn_bwd_host, *bad)
        assert code == -2 and "lse" in msg
    # an output on the wrong side, and a device buffer that is not on the device
    code, msg = _code(ab.attn_bwd_host, *t, dq=torch.empty(B, S, HQ, D, dtype=torch.bfloat16,
                                                             device="meta"))
    assert code == -9 and "dq" in msg
    code, msg = _code(ab.attn_bwd_host, *t, device_buffer=torch.empty(16, dtype=torch.uint8))
    assert code == -9 and "device_buffer" in msg


def test_host_varlen_checks_packed_shapes():
    tq, tk = 100, 80
    q = torch.randn(tq, HQ, D).to(torch.bfloat16)
    k = torch.randn(tk, HK, D).to(torch.bfloat16)
    v = torch.randn(tk, HK, D).to(torch.bfloat16)
    cu_q = torch.tensor([0, 40, 100], dtype=torch.int32)
    cu_k = torch.tensor([0, 30, 80], dtype=torch.int32)
    # LSE of a packed call is [H_q, total_q]; the padded [B, H_q, S] layout is refused
    code, msg = _code(ab.attn_bwd_host_varlen, q, k, v, q.clone(), torch.zeros(1, HQ, tq),
                      q.clone(), cu_q, cu_k)
    assert code == -2 and "lse" in msg
    # padded tensors given to the packed entry point
    code, _ = _code(ab.attn_bwd_host_varlen, q[None], k[None], v[None], q[None],
                    torch.zeros(HQ, tq), q[None], cu_q, cu_k)
    assert code == -2
