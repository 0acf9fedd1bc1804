"""attn_bwd_host (tensors in host memory, chunked and overlapped copies)
against attn_bwd on the same data on the device, and once against the oracle.

Each chunk of attn_bwd_host is an independent backward problem, so dK and dV
(computed by one CTA per key tile, no atomics) must come out bit for bit as
attn_bwd's, and so must dQ in deterministic mode; otherwise dQ's fp32 adds may
land in another order and dQ is compared within the parity tolerance.
"""
import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _pinned(t):
    return t.contiguous().pin_memory()


def _problem(b, hq, hk, sq, sk, d, dtype, causal, seed):
    w = synth.small("host", b, hq, hk, sq, sk, d, dtype, causal, seed)
    x = synth.make_inputs(w)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    o, lse = ab.attn_fwd(q, k, v, causal=causal)
    return w, x, (q, k, v, o, lse, do)


def _compare(dev, host, deterministic, name):
    for tag, g, r in zip(("dQ", "dK", "dV"), host, dev):
        if tag != "dQ" or deterministic:
            assert torch.equal(g, r.cpu()), f"{name} {tag} differs from attn_bwd"
        else:
            # a reordered fp32 sum can move an element across a rounding boundary of
            # the 16-bit output: at most one unit in the last place (< 2^-7 relative)
            assert_close(f"{name} {tag}", g, r.float().cpu().double().numpy(), rel_l2=1e-3,
                         max_frac=1e-2)


CASES = [
    # B, Hq, Hk, Sq, Sk, D, dtype, causal, chunks
    (2, 8, 2, 700, 700, 128, "bf16", True, 0),     # auto: one sequence x one kv head per chunk
    (2, 8, 2, 700, 700, 128, "bf16", True, 1),     # one chunk: the whole problem
    (2, 8, 2, 700, 700, 128, "bf16", True, 2),     # one sequence per chunk
    (5, 4, 4, 300, 300, 64, "fp16", False, 2),     # runs of 3 and 2 sequences
    (1, 16, 4, 513, 1000, 128, "bf16", True, 4),   # Sq < Sk, four kv-head chunks
    (3, 6, 3, 257, 129, 64, "bf16", True, 9),      # one kv head per chunk, Sq > Sk
    (2, 4, 2, 300, 300, 96, "bf16", True, 0),      # D = 96 tiles
    (1, 4, 2, 257, 257, 192, "bf16", True, 2),     # D = 192: two passes on three-chunk tiles
    (2, 2, 1, 200, 200, 256, "fp16", False, 0),    # D = 256
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}h{c[1]}k{c[2]}s{c[3]}x{c[4]}d{c[5]}c{c[8]}"
                                             for c in CASES])
def test_host_matches_device(case):
    b, hq, hk, sq, sk, d, dtype, causal, chunks = case
    w, x, (q, k, v, o, lse, do) = _problem(b, hq, hk, sq, sk, d, dtype, causal, 31 + sum(case[:5]))
    dev = ab.attn_bwd(q, k, v, o, lse, do, causal=causal)
    host_in = [_pinned(t.cpu()) for t in (q, k, v, o, lse, do)]
    got = ab.attn_bwd_host(*host_in, causal=causal, chunks=chunks)
    torch.cuda.synchronize()
    ab.check_device_status()
    _compare(dev, got, False, w.name)


@pytest.mark.parametrize("chunks", [0, 3])
def test_host_deterministic_bit_exact(chunks):
    w, x, (q, k, v, o, lse, do) = _problem(2, 8, 2, 640, 640, 128, "bf16", True, 5)
    dev = ab.attn_bwd(q, k, v, o, lse, do, causal=True, deterministic=True)
    host_in = [_pinned(t.cpu()) for t in (q, k, v, o, lse, do)]
    got = ab.attn_bwd_host(*host_in, causal=True, deterministic=True, chunks=chunks)
    torch.cuda.synchronize()
    ab.check_device_status()
    _compare(dev, got, True, w.name)


def test_host_strided_tensors_and_oracle():
    """Host tensors whose positions are padded (stride_s > H*D), results
    checked against the fp64 oracle; the output tensors are padded too."""
    b, hq, hk, s, d = 2, 4, 2, 400, 128
    w, x, (q, k, v, o, lse, do) = _problem(b, hq, hk, s, s, d, "bf16", True, 77)

    def padded(t):
        big = torch.zeros(t.shape[0], t.shape[1], t.shape[2] + 1, t.shape[3], dtype=t.dtype,
                          pin_memory=True)
        big[:, :, : t.shape[2]] = t.cpu()
        return big[:, :, : t.shape[2]]

    hin = [padded(t) for t in (q, k, v, o)]
    hdo = padded(do)
    outs = [padded(torch.full_like(t, float("nan"))) for t in (q, k, v)]
    got = ab.attn_bwd_host(*hin, _pinned(lse.cpu()), hdo, *outs, causal=True, chunks=0)
    torch.cuda.synchronize()
    ab.check_device_status()
    assert got[0].stride(1) == (hq + 1) * d
    ref = attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, True, None, None)
    floor = float(np.abs(ref["dV"]).max())
    for name, g in zip(("dQ", "dK", "dV"), got):
        assert_close(f"host strided {name}", g, ref[name], floor=floor)


@pytest.mark.parametrize("sq,sk", [(0, 200), (200, 0)])
def test_host_empty_sides(sq, sk):
    b, hq, hk, d = 2, 4, 2, 64
    dt = torch.bfloat16
    q = torch.randn(b, sq, hq, d, dtype=dt).pin_memory()
    o = torch.randn(b, sq, hq, d, dtype=dt).pin_memory()
    do = torch.randn(b, sq, hq, d, dtype=dt).pin_memory()
    k = torch.randn(b, sk, hk, d, dtype=dt).pin_memory()
    v = torch.randn(b, sk, hk, d, dtype=dt).pin_memory()
    lse = torch.zeros(b, hq, sq).pin_memory()
    dq = torch.full_like(q, float("nan")).pin_memory()
    dk = torch.full_like(k, float("nan")).pin_memory()
    dv = torch.full_like(v, float("nan")).pin_memory()
    ab.attn_bwd_host(q, k, v, o, lse, do, dq, dk, dv, causal=False)
    torch.cuda.synchronize()
    ab.check_device_status()
    for t in (dq, dk, dv):
        assert not t.isnan().any() and (t == 0).all()


def test_host_two_calls_reuse_buffer_and_stream_order():
    """Two calls back to back on one stream with one device buffer: the second
    starts only after the first has finished with the buffer."""
    w, x, (q, k, v, o, lse, do) = _problem(2, 8, 4, 500, 500, 128, "bf16", False, 9)
    dev = ab.attn_bwd(q, k, v, o, lse, do, causal=False, deterministic=True)
    buf = torch.empty(ab.host_buffer_size(2, 500, 500, 8, 4, 128, 0), dtype=torch.uint8,
                      device="cuda")
    host_in = [_pinned(t.cpu()) for t in (q, k, v, o, lse, do)]
    outs = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, k, v)]
            for _ in range(2)]
    for out in outs:
        ab.attn_bwd_host(*host_in, *out, causal=False, deterministic=True, device_buffer=buf)
    torch.cuda.synchronize()
    ab.check_device_status()
    for out in outs:
        _compare(dev, out, True, "two calls")


def test_host_with_window_and_softcap():
    """attn_opts pass through the host pipeline: a sliding window and a logit cap
    give attn_bwd's results (deterministic mode: bit for bit)."""
    w, x, (q, k, v, o, lse, do) = _problem(2, 8, 2, 700, 700, 128, "bf16", True, 13)
    o, lse = ab.attn_fwd(q, k, v, causal=True, window=(200, -1), softcap=3.0)
    dev = ab.attn_bwd(q, k, v, o, lse, do, causal=True, deterministic=True, window=(200, -1),
                      softcap=3.0)
    host_in = [_pinned(t.cpu()) for t in (q, k, v, o, lse, do)]
    got = ab.attn_bwd_host(*host_in, causal=True, deterministic=True, window=(200, -1),
                           softcap=3.0)
    torch.cuda.synchronize()
    ab.check_device_status()
    _compare(dev, got, True, "host window softcap")


@pytest.mark.parametrize("det,window,chunks", [(False, None, 0), (True, None, 3),
                                               (False, (64, 16), 2)])
def test_host_varlen_matches_device(det, window, chunks):
    """Packed sequences (empty ones, cross attention with cu_seqlens_q !=
    cu_seqlens_k) through attn_bwd_host_varlen: equal to attn_bwd's results."""
    lq, lk = [300, 0, 17, 640, 129, 5], [200, 150, 0, 513, 129, 5]
    w = synth.Workload("hostvl", 0, 8, 2, 0, 0, 128, "bf16", window is None, 71, n_seqs=len(lq),
                       len_lo=0, len_hi=700)
    x = synth.make_inputs(w, lengths=lq, lengths_k=lk)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    kw = dict(cu_seqlens_q=x.cu_seqlens_q.cuda(), cu_seqlens_k=x.cu_seqlens_k.cuda(),
              max_seqlen_q=max(lq), max_seqlen_k=max(lk), causal=w.causal, window=window)
    o, lse = ab.attn_fwd(q, k, v, **kw)
    dev = ab.attn_bwd(q, k, v, o, lse, do, deterministic=det, **kw)
    host_in = [_pinned(t.cpu()) for t in (q, k, v, o, lse, do)]
    got = ab.attn_bwd_host_varlen(*host_in, x.cu_seqlens_q, x.cu_seqlens_k, causal=w.causal,
                                  deterministic=det, chunks=chunks, window=window)
    torch.cuda.synchronize()
    ab.check_device_status()
    _compare(dev, got, det, "host varlen")
