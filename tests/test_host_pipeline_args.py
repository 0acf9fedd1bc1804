"""Host-side checks of attn_bwd_host and attn_bwd_host_buffer_size (no GPU
needed): the buffer size follows the chunking, and bad arguments are rejected
with the documented status codes before anything is enqueued."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from attention_backward_bwd_gb300 import binding
    return binding.lib()


def _t(ptr, b, s, h, d, stride_s=None, stride_h=None):
    from attention_backward_bwd_gb300.binding import AttnTensor
    ss = h * d if stride_s is None else stride_s
    return AttnTensor(ptr, s * ss, ss, d if stride_h is None else stride_h)


def _call(lib, b=2, sq=256, sk=256, hq=8, hk=2, d=128, dtype=1, chunks=0, buf=1 << 24,
          buf_bytes=None, q_stride_h=None, q_ptr=1 << 20, lse=1 << 21):
    q = _t(q_ptr, b, sq, hq, d, stride_h=q_stride_h)
    qo = _t(1 << 20, b, sq, hq, d)
    k = _t(1 << 20, b, sk, hk, d)
    if buf_bytes is None:
        buf_bytes = lib.attn_bwd_host_buffer_size(b, sq, sk, hq, hk, d, chunks)
    return lib.attn_bwd_host(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), ctypes.byref(qo),
                             lse, ctypes.byref(qo), ctypes.byref(qo), ctypes.byref(k),
                             ctypes.byref(k), dtype, b, sq, sk, hq, hk, d, 0.1, 1, 0, None, chunks,
                             buf, buf_bytes, None)


def test_buffer_size_covers_tensors_and_follows_chunks(lib):
    b, s, hq, hk, d = 2, 8192, 32, 8, 128
    tensors = 4 * b * s * hq * d * 2 + 4 * b * s * hk * d * 2 + b * hq * s * 4
    whole = lib.attn_bwd_host_buffer_size(b, s, s, hq, hk, d, 1)
    auto = lib.attn_bwd_host_buffer_size(b, s, s, hq, hk, d, 0)
    eight = lib.attn_bwd_host_buffer_size(b, s, s, hq, hk, d, 8)
    assert auto == eight  # the library's default is 8 chunks
    assert tensors < auto < whole  # smaller chunks, smaller workspaces
    ws_whole = lib.attn_bwd_workspace_size(b, s, hq, d, 0, 0)
    assert whole >= tensors + 3 * ws_whole  # one workspace per compute stream
    assert lib.attn_bwd_host_buffer_size(0, s, s, hq, hk, d, 0) == 0
    assert lib.attn_bwd_host_buffer_size(b, s, s, 6, 4, d, 0) == 0  # h_q % h_k != 0


@pytest.mark.parametrize("case,code", [
    ("dtype", -1), ("head_dim", -2), ("gqa_ratio", -2), ("heads_not_adjacent", -3),
    ("null_q", -5), ("null_lse", -5), ("null_buffer", -6), ("small_buffer", -6),
    ("buffer_align", -6),
])
def test_argument_errors(lib, case, code):
    kw = {}
    if case == "dtype":
        kw["dtype"] = 7
    elif case == "head_dim":
        kw["d"] = 100  # not a multiple of 8
    elif case == "gqa_ratio":
        kw.update(hq=6, hk=4)
    elif case == "heads_not_adjacent":
        kw["q_stride_h"] = 256
    elif case == "null_q":
        kw["q_ptr"] = None
    elif case == "null_lse":
        kw["lse"] = None
    elif case == "null_buffer":
        kw["buf"] = None
    elif case == "small_buffer":
        kw["buf_bytes"] = 1 << 20
    elif case == "buffer_align":
        kw["buf"] = (1 << 24) + 128
    rc = _call(lib, **kw)
    assert rc == code, (rc, lib.attn_last_error())
    assert lib.attn_last_error()


def test_bad_options_rejected(lib):
    from attention_backward_bwd_gb300.binding import AttnOpts
    q = _t(1 << 20, 2, 256, 8, 128)
    k = _t(1 << 20, 2, 256, 2, 128)
    opts = AttnOpts(-2, 0, 0.0)
    size = lib.attn_bwd_host_buffer_size(2, 256, 256, 8, 2, 128, 0)
    rc = lib.attn_bwd_host(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), ctypes.byref(q),
                           1 << 21, ctypes.byref(q), ctypes.byref(q), ctypes.byref(k),
                           ctypes.byref(k), 1, 2, 256, 256, 8, 2, 128, 0.1, 1, 0,
                           ctypes.byref(opts), 0, 1 << 24, size, None)
    assert rc == -9 and b"window" in lib.attn_last_error()


def test_varlen_buffer_size_and_bad_cu(lib):
    import numpy as np
    cu = np.array([0, 300, 300, 1000, 1500], dtype=np.int32)
    size = lib.attn_bwd_host_varlen_buffer_size(cu.ctypes.data, cu.ctypes.data, 4, 1500, 1500, 8,
                                                2, 128, 0)
    tensors = 4 * 1500 * 8 * 128 * 2 + 4 * 1500 * 2 * 128 * 2 + 8 * 1500 * 4
    assert size > tensors and size % 256 == 0
    for bad, msg in (([0, 300, 200, 1000, 1500], b"nondecreasing"),
                     ([1, 300, 300, 1000, 1500], b"start at 0"),
                     ([0, 300, 300, 1000, 1499], b"end at")):
        arr = np.array(bad, dtype=np.int32)
        assert lib.attn_bwd_host_varlen_buffer_size(arr.ctypes.data, cu.ctypes.data, 4, 1500, 1500,
                                                    8, 2, 128, 0) == 0
        assert msg in lib.attn_last_error()


def test_seqused_refused_by_the_host_calls(lib):
    """Used lengths are device arrays read by the kernels; the host-buffer calls
    take host tensors, so they refuse seqused_q/k rather than hand a kernel a
    pointer of the wrong kind."""
    import numpy as np
    from attention_backward_bwd_gb300.binding import AttnOpts
    used = np.array([100, 200], dtype=np.int32)
    q = _t(1 << 20, 2, 256, 8, 128)
    k = _t(1 << 20, 2, 256, 2, 128)
    for opts in (AttnOpts(-1, -1, 0.0, used.ctypes.data, None),
                 AttnOpts(-1, -1, 0.0, None, used.ctypes.data)):
        size = lib.attn_bwd_host_buffer_size(2, 256, 256, 8, 2, 128, 0)
        rc = lib.attn_bwd_host(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k),
                               ctypes.byref(q), 1 << 21, ctypes.byref(q), ctypes.byref(q),
                               ctypes.byref(k), ctypes.byref(k), 1, 2, 256, 256, 8, 2, 128, 0.1,
                               1, 0, ctypes.byref(opts), 0, 1 << 24, size, None)
        assert rc == -9 and b"seqused" in lib.attn_last_error()
        cu = np.array([0, 200, 512], dtype=np.int32)
        pq = _t(1 << 20, 1, 512, 8, 128)
        pk = _t(1 << 20, 1, 512, 2, 128)
        vsize = lib.attn_bwd_host_varlen_buffer_size(cu.ctypes.data, cu.ctypes.data, 2, 512, 512,
                                                     8, 2, 128, 0)
        rc = lib.attn_bwd_host_varlen(ctypes.byref(pq), ctypes.byref(pk), ctypes.byref(pk),
                                      ctypes.byref(pq), 1 << 21, ctypes.byref(pq),
                                      ctypes.byref(pq), ctypes.byref(pk), ctypes.byref(pk), 1, 2,
                                      512, 512, 8, 2, 128, 0.1, 1, cu.ctypes.data, cu.ctypes.data,
                                      0, ctypes.byref(opts), 0, 1 << 24, vsize, None)
        assert rc == -9 and b"seqused" in lib.attn_last_error()
