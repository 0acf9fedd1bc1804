"""GPU backward (attn_bwd through the C ABI) against the fp64 CPU oracle.

Primary check: GPU attn_fwd -> GPU attn_bwd, compared with the all-fp64
oracle gradients of the same rounded inputs.  Secondary check: the oracle's
O (rounded to the dtype) and LSE are fed to the GPU backward, isolating the
backward's own error.  Tolerance: rel-L2 <= 1e-2, max-abs <= 2e-2 * max|ref|.
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

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def run_gpu(w, x, deterministic=False, o=None, lse=None):
    (q, k, v, do), cu_q, cu_k = to_dev(x)
    mq = mk = None
    if cu_q is not None:
        mq = max(x.lengths) if x.lengths else 0
        mk = max(x.lengths_k) if x.lengths_k else 0
    if o is None:
        o, lse = ab.attn_fwd(q, k, v, causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                             max_seqlen_q=mq, max_seqlen_k=mk)
    dq, dk, dv = ab.attn_bwd(q, k, v, o, lse, do, causal=w.causal, cu_seqlens_q=cu_q,
                             cu_seqlens_k=cu_k, max_seqlen_q=mq, max_seqlen_k=mk,
                             deterministic=deterministic or w.deterministic)
    ab.check_device_status()
    return dq, dk, dv


def oracle_grads(w, x):
    return attn_oracle.mha_backward(x.q, x.k, x.v, x.do, w.scale, w.causal, x.cu_seqlens_q,
                                    x.cu_seqlens_k)


def check(w, x, deterministic=False):
    dq, dk, dv = run_gpu(w, x, deterministic)
    ref = oracle_grads(w, x)
    out = {}
    floor = float(np.abs(ref["dV"]).max())
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        out[name] = assert_close(f"{w.name} {name}", got, ref[name], floor=floor)
    return out


@pytest.mark.parametrize("name", ["mha_b1_h2_s128_d64_fp16", "mha_b4_h16_s1024_d64_fp16_causal"])
def test_small_workloads_full(name):
    w = synth.WORKLOADS[name]
    check(w, synth.make_inputs(w))


EDGE = [
    # B, Hq, Hk, Sq, Sk, D, dtype, causal
    (1, 1, 1, 1, 1, 64, "bf16", False),
    (1, 2, 2, 63, 63, 64, "fp16", True),
    (1, 2, 1, 65, 65, 128, "bf16", True),
    (2, 2, 2, 129, 129, 128, "fp16", False),
    (1, 4, 2, 200, 200, 64, "bf16", True),
    (2, 4, 1, 300, 300, 128, "bf16", True),
    (1, 2, 2, 256, 256, 128, "bf16", False),
    (1, 2, 2, 100, 300, 128, "bf16", False),  # Sq < Sk
    (1, 2, 2, 100, 300, 64, "fp16", True),    # causal, bottom-right alignment
    (1, 2, 2, 300, 100, 128, "bf16", True),   # causal Sq > Sk: leading rows see no key
    (1, 8, 2, 384, 384, 128, "bf16", True),   # GQA 4:1, several tiles
    (1, 8, 1, 520, 520, 128, "bf16", True),   # GQA 8:1, ragged last tile
    (2, 4, 2, 257, 700, 64, "bf16", True),    # causal Sq < Sk, D=64 GQA, ragged both sides
    (1, 4, 4, 640, 333, 128, "fp16", True),   # causal Sq > Sk over several query tiles
    (1, 2, 2, 1000, 1000, 128, "fp16", False),  # fp16, 8 tiles, ragged
]


@pytest.mark.parametrize("case", EDGE, ids=str)
def test_edge_shapes(case):
    b, hq, hk, sq, sk, d, dtype, causal = case
    w = synth.small("edge", b, hq, hk, sq, sk, d, dtype, causal, 50 + sq + sk)
    check(w, synth.make_inputs(w))


@pytest.mark.parametrize("case", EDGE[3:7] + EDGE[-4:-1], ids=str)
def test_edge_shapes_deterministic(case):
    b, hq, hk, sq, sk, d, dtype, causal = case
    w = synth.small("edge_det", b, hq, hk, sq, sk, d, dtype, causal, 60 + sq, deterministic=True)
    check(w, synth.make_inputs(w), deterministic=True)


def test_secondary_oracle_forward_inputs():
    w = synth.small("sec", 2, 4, 2, 333, 333, 128, "bf16", True, 71)
    x = synth.make_inputs(w)
    o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, True)
    o = torch.tensor(o_ref).to(torch.bfloat16).cuda()
    lse = torch.tensor(lse_ref, dtype=torch.float32).cuda()
    dq, dk, dv = run_gpu(w, x, o=o, lse=lse)
    ref = oracle_grads(w, x)
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert_close(name, got, ref[name])


def test_varlen_with_empty_sequences():
    lens = [5, 130, 0, 64, 1, 257, 128]
    w = synth.Workload("vl", 0, 4, 2, 0, 0, 128, "bf16", True, 81, n_seqs=len(lens), len_lo=0,
                       len_hi=300)
    check(w, synth.make_inputs(w, lengths=lens))


def test_varlen_deterministic_d64():
    lens = [300, 17, 129]
    w = synth.Workload("vl64", 0, 2, 2, 0, 0, 64, "fp16", False, 82, n_seqs=3, len_lo=1,
                       len_hi=300, deterministic=True)
    check(w, synth.make_inputs(w, lengths=lens), deterministic=True)


CROSS = [
    # query lengths, key lengths, Hq, Hk, D, dtype, causal, deterministic
    ([300, 0, 17, 129, 5, 640], [200, 150, 0, 513, 5, 64], 4, 2, 128, "bf16", True, False),
    ([300, 0, 17, 129, 5, 640], [200, 150, 0, 513, 5, 64], 4, 2, 128, "bf16", False, False),
    ([1000, 64, 0, 257], [257, 700, 333, 0], 2, 2, 64, "fp16", True, False),
    ([300, 0, 17, 129, 5, 640], [200, 150, 0, 513, 5, 64], 8, 2, 128, "bf16", True, True),
]


@pytest.mark.parametrize("case", CROSS, ids=[f"cross{i}" for i in range(len(CROSS))])
def test_cross_attention_varlen(case):
    """Packed sequences whose query and key lengths differ (cu_seqlens_q !=
    cu_seqlens_k): causal masks align bottom-right per sequence, a sequence
    with keys but no queries gets dK = dV = 0 exactly, one with queries but no
    keys gets dQ = 0.  Outputs start as NaN so an unwritten row shows."""
    lq, lk, hq, hk, d, dt, causal, det = case
    w = synth.Workload("cross", 0, hq, hk, 0, 0, d, dt, causal, 83 + len(lq), n_seqs=len(lq),
                       len_lo=0, len_hi=1000, deterministic=det)
    x = synth.make_inputs(w, lengths=lq, lengths_k=lk)
    (q, k, v, do), cu_q, cu_k = to_dev(x)
    mq, mk = max(lq), max(lk)
    o, lse = ab.attn_fwd(q, k, v, causal=causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                         max_seqlen_q=mq, max_seqlen_k=mk)
    runs = []
    for _ in range(2 if det else 1):
        outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        ab.attn_bwd(q, k, v, o, lse, do, causal=causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                    max_seqlen_q=mq, max_seqlen_k=mk, deterministic=det, dq=outs[0],
                    dk=outs[1], dv=outs[2])
        ab.check_device_status()
        runs.append(outs)
    if det:
        for a, b in zip(*runs):
            assert torch.equal(a, b)
    dq, dk, dv = runs[0]
    for t in (dq, dk, dv):
        assert not t.isnan().any()
    cq, ck = np.cumsum([0] + lq), np.cumsum([0] + lk)
    for b in range(len(lq)):
        if lq[b] == 0:
            assert (dk[ck[b]:ck[b + 1]] == 0).all() and (dv[ck[b]:ck[b + 1]] == 0).all()
        if lk[b] == 0:
            assert (dq[cq[b]:cq[b + 1]] == 0).all()
    ref = oracle_grads(w, x)
    floor = float(np.abs(ref["dV"]).max())
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert_close(f"cross {name}", got, ref[name], floor=floor)


HEAD_DIMS = [
    # B, Hq, Hk, Sq, Sk, D, dtype, causal: D below 64 runs on the D = 64 kernel, in
    # (64, 96] on the D = 96 kernel, in (96, 128) on the D = 128 one, with the extra
    # head-dimension columns zero
    (1, 4, 2, 300, 300, 32, "bf16", True),
    (2, 2, 2, 257, 257, 48, "fp16", False),
    (1, 4, 4, 513, 513, 80, "bf16", True),
    (1, 8, 2, 700, 700, 96, "bf16", True),
    (2, 2, 2, 257, 257, 88, "fp16", False),
    (1, 2, 2, 1000, 1000, 96, "fp16", True),
    (1, 2, 1, 200, 333, 112, "bf16", False),
    (1, 2, 2, 129, 129, 8, "bf16", True),
]


@pytest.mark.parametrize("case", HEAD_DIMS, ids=[f"d{c[5]}" for c in HEAD_DIMS])
def test_padded_head_dims(case):
    b, hq, hk, sq, sk, d, dt, causal = case
    w = synth.small(f"d{d}", b, hq, hk, sq, sk, d, dt, causal, 500 + d)
    check(w, synth.make_inputs(w))


def test_padded_head_dim_deterministic_varlen():
    lens = [300, 0, 129, 640]
    w = synth.Workload("d96vl", 0, 8, 2, 0, 0, 96, "bf16", True, 597, n_seqs=len(lens),
                       len_lo=0, len_hi=700, deterministic=True)
    x = synth.make_inputs(w, lengths=lens)
    runs = [run_gpu(w, x, deterministic=True) for _ in range(2)]
    for a, r in zip(*runs):
        assert torch.equal(a, r)
    ref = oracle_grads(w, x)
    for name, got in zip(("dQ", "dK", "dV"), runs[0]):
        assert_close(f"d96 varlen {name}", got, ref[name])


def test_deterministic_is_bitwise_repeatable():
    w = synth.small("det", 1, 8, 2, 1000, 1000, 128, "bf16", True, 91, deterministic=True)
    x = synth.make_inputs(w)
    runs = [run_gpu(w, x, deterministic=True) for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    ref = oracle_grads(w, x)
    for name, got in zip(("dQ", "dK", "dV"), runs[0]):
        assert_close(name, got, ref[name])


def test_empty_query_and_key_sides():
    (q, k, v, do) = [torch.randn(1, 0, 2, 64, dtype=torch.bfloat16, device="cuda")
                     for _ in range(4)]
    k = torch.randn(1, 50, 2, 64, dtype=torch.bfloat16, device="cuda")
    v = torch.randn_like(k)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 0, device="cuda")
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    ab.attn_bwd(q, k, v, o, lse, do, dk=dk, dv=dv)
    ab.check_device_status()
    assert (dk == 0).all() and (dv == 0).all()
    q = torch.randn(1, 40, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(1, 0, 2, 64, dtype=torch.bfloat16, device="cuda")
    dq = torch.full_like(q, 7.0)
    ab.attn_bwd(q, k, k, q, torch.zeros(1, 2, 40, device="cuda"), q, dq=dq)
    ab.check_device_status()
    assert (dq == 0).all()


def test_strided_inputs():
    """Heads taken from a wider tensor: stride_h = D, stride_s = 2*H*D."""
    w = synth.small("str", 2, 4, 2, 160, 160, 64, "bf16", False, 93)
    x = synth.make_inputs(w)
    dev = "cuda"

    def widen(t):
        big = torch.zeros(t.shape[0], t.shape[1], 2 * t.shape[2], t.shape[3], dtype=t.dtype)
        big[:, :, 1::2] = t
        return big.to(dev)[:, :, 1::2]

    q, k, v, do = (widen(t) for t in (x.q, x.k, x.v, x.do))
    assert q.stride(2) == 2 * 64
    o, lse = ab.attn_fwd(q, k, v)
    dq, dk, dv = ab.attn_bwd(q, k, v, o, lse, do)
    ab.check_device_status()
    ref = oracle_grads(w, x)
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert_close(name, got, ref[name])


def test_full_size_invariants_mha_s1024():
    """Properties that hold at any size: sum_j dV_j = sum_i dO_i per head
    (rows of P sum to one) and sum_j dK_j = 0 per kv head (rows of dS sum to 0)."""
    w = synth.WORKLOADS["mha_b4_h16_s1024_d64_fp16_causal"]
    x = synth.make_inputs(w)
    dq, dk, dv = run_gpu(w, x)
    sdv = dv.double().sum(dim=1).cpu()
    sdo = x.do.double().sum(dim=1)
    assert torch.allclose(sdv, sdo, rtol=2e-2, atol=2e-2 * sdo.abs().max().item())
    sdk = dk.double().sum(dim=1).cpu()
    assert sdk.abs().max().item() <= 2e-2 * dk.double().abs().sum(dim=1).max().item()


def test_full_size_bench_workload_sampled_rows():
    """The benchmark's own workload at full size (GQA B=2, Hq=32, Hk=8, S=8192,
    D=128, bf16, causal) through the same calls bench.py times.  dQ at sampled
    query rows and dK, dV at sampled key rows of two (sequence, kv head) groups
    are compared with the fp64 oracle evaluated row by row (tile boundaries,
    first and last rows, and random rows)."""
    w = synth.WORKLOADS["gqa_b2_hq32_hk8_s8192_d128_bf16_causal"]
    x = synth.make_inputs(w)
    dq, dk, dv = run_gpu(w, x)
    rng = np.random.default_rng(2024)
    rows = sorted(set([0, 1, 127, 128, 129, 4095, 4096, 8064, 8190, 8191] +
                      [int(r) for r in rng.integers(0, w.seqlen_q, 6)]))
    grp = w.h_q // w.h_k
    for b, g in ((0, 0), (1, 5)):
        dq_ref, dk_ref, dv_ref = attn_oracle.group_backward_rows(x.q, x.k, x.v, x.do, b, g, rows,
                                                                 rows, w.scale, w.causal)
        got_dq = dq[b, rows, g * grp:(g + 1) * grp].transpose(0, 1)
        assert_close(f"full-size dQ b={b} g={g}", got_dq, dq_ref)
        assert_close(f"full-size dK b={b} g={g}", dk[b, rows, g], dk_ref)
        assert_close(f"full-size dV b={b} g={g}", dv[b, rows, g], dv_ref)


@pytest.mark.parametrize("name", ["gqa_b2_hq32_hk8_s8192_d128_bf16_causal_win1024",
                                  "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_cap30"])
def test_full_size_window_and_softcap_sampled_rows(name):
    """The sliding-window and logit-cap bench workloads at full size, through
    the options bench.py passes, on sampled rows (including rows around the
    window's edge) of one group against the row-wise fp64 oracle."""
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.do))
    window = tuple(w.window) if w.windowed else None
    o, lse = ab.attn_fwd(q, k, v, causal=w.causal, window=window, softcap=w.softcap)
    dq, dk, dv = ab.attn_bwd(q, k, v, o, lse, do, causal=w.causal, window=window,
                             softcap=w.softcap)
    ab.check_device_status()
    rng = np.random.default_rng(11)
    rows = sorted(set(_sampled_rows(w.seqlen_q, rng) + [1023, 1024, 1025, 1151, 1152, 5000]))
    grp = w.h_q // w.h_k
    b, g = 1, 3
    dq_ref, dk_ref, dv_ref = attn_oracle.group_backward_rows(
        x.q, x.k, x.v, x.do, b, g, rows, rows, w.scale, w.causal, window=window,
        softcap=w.softcap)
    assert_close(f"{name} dQ", dq[b, rows, g * grp:(g + 1) * grp].transpose(0, 1), dq_ref)
    assert_close(f"{name} dK", dk[b, rows, g], dk_ref)
    assert_close(f"{name} dV", dv[b, rows, g], dv_ref)


def _sampled_rows(n, rng, extra=6):
    base = [0, 1, 127, 128, 129, n // 2, n - 2, n - 1]
    return sorted(set(r for r in base + [int(v) for v in rng.integers(0, n, extra)] if 0 <= r < n))


@pytest.mark.parametrize("name", ["mha_b2_h16_s4096_d128_bf16", "mha_b2_h16_s4096_d128_bf16_causal",
                                  "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_det"])
def test_full_size_configs_sampled_rows(name):
    """The other padded benchmark configs at full size, through the calls bench.py
    times, on sampled rows of one (sequence, kv head) group against the row-wise
    fp64 oracle; the deterministic config is also checked bit for bit against a
    second run."""
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    dq, dk, dv = run_gpu(w, x)
    rng = np.random.default_rng(7)
    rows = _sampled_rows(w.seqlen_q, rng)
    grp = w.h_q // w.h_k
    b, g = w.batch - 1, w.h_k - 1
    dq_ref, dk_ref, dv_ref = attn_oracle.group_backward_rows(x.q, x.k, x.v, x.do, b, g, rows, rows,
                                                             w.scale, w.causal)
    assert_close(f"{name} dQ", dq[b, rows, g * grp:(g + 1) * grp].transpose(0, 1), dq_ref)
    assert_close(f"{name} dK", dk[b, rows, g], dk_ref)
    assert_close(f"{name} dV", dv[b, rows, g], dv_ref)
    if w.deterministic:
        dq2, dk2, dv2 = run_gpu(w, x)
        assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_full_size_varlen_sampled_rows():
    """The varlen config at full size (16 packed sequences, lengths drawn from
    [128, 8192]); the shortest and the longest sequence are checked on sampled
    rows of one head each against the row-wise fp64 oracle on that sequence."""
    w = synth.WORKLOADS["varlen16_h16_d128_bf16_causal"]
    x = synth.make_inputs(w)
    dq, dk, dv = run_gpu(w, x)
    cu = [int(c) for c in x.cu_seqlens_q]
    lens = x.lengths
    rng = np.random.default_rng(11)
    for bsel, h in ((int(np.argmin(lens)), 3), (int(np.argmax(lens)), 12)):
        lo, hi = cu[bsel], cu[bsel + 1]
        rows = _sampled_rows(hi - lo, rng)
        seq = [t[lo:hi].unsqueeze(0) for t in (x.q, x.k, x.v, x.do)]
        dq_ref, dk_ref, dv_ref = attn_oracle.group_backward_rows(*seq, 0, h, rows, rows, w.scale,
                                                                 w.causal)
        idx = [lo + r for r in rows]
        assert_close(f"varlen seq {bsel} dQ", dq[idx, h].unsqueeze(0), dq_ref)
        assert_close(f"varlen seq {bsel} dK", dk[idx, h], dk_ref)
        assert_close(f"varlen seq {bsel} dV", dv[idx, h], dv_ref)


_LONG = synth.small("long", 1, 2, 1, 32768, 32768, 128, "bf16", True, 4242)


@functools.lru_cache(maxsize=1)
def _long_case():
    """Inputs and row-wise oracle gradients of the long-sequence case, computed
    once for both of its tests (the oracle takes about a minute on the host)."""
    x = synth.make_inputs(_LONG)
    rng = np.random.default_rng(5)
    rows = sorted(set(_sampled_rows(_LONG.seqlen_q, rng) + [16383, 16384, 32640]))
    refs = attn_oracle.group_backward_rows(x.q, x.k, x.v, x.do, 0, 0, rows, rows, _LONG.scale,
                                           _LONG.causal)
    return x, rows, refs


@pytest.mark.parametrize("deterministic", [False, True], ids=["nondet", "det"])
def test_long_sequence_sampled_rows(deterministic):
    """One long sequence, S = 32768 (256 key tiles; the unit of key tile 0 runs
    512 tiles, and in deterministic mode a query tile's adds form a chain of up
    to 256 key tiles), GQA 2:1, D = 128, bf16, causal: sampled rows against the
    row-wise fp64 oracle; deterministic mode also bit for bit against a second
    run."""
    x, rows, (dq_ref, dk_ref, dv_ref) = _long_case()
    dq, dk, dv = run_gpu(_LONG, x, deterministic)
    assert_close("long dQ", dq[0, rows, 0:2].transpose(0, 1), dq_ref)
    assert_close("long dK", dk[0, rows, 0], dk_ref)
    assert_close("long dV", dv[0, rows, 0], dv_ref)
    if deterministic:
        dq2, dk2, dv2 = run_gpu(_LONG, x, deterministic)
        assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
