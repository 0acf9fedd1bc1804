"""GPU forward (attn_fwd through the C ABI) against the fp64 oracle's O and LSE.

The forward produces the O and the natural-log LSE the backward consumes
(TileLang test_tilelang_kernel_mha_bwd.py, flashattn_fwd).  Tolerance on O:
the stated rel-L2 <= 1e-2 and max-abs <= 2e-2 * max|ref|; LSE to 2e-3
absolute; rows without an allowed key must give O = 0 and LSE = +inf.
"""
import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _check(o, lse, o_ref, lse_ref, tag):
    assert_close(f"{tag} O", o, o_ref)
    lc = lse.cpu().double().numpy()
    fin = np.isfinite(lse_ref)
    assert (np.isinf(lc) == ~fin).all(), f"{tag}: rows without keys"
    assert (lc[~fin] > 0).all()
    np.testing.assert_allclose(lc[fin], lse_ref[fin], rtol=0, atol=2e-3, err_msg=tag)
    o_rows = o.float().cpu().numpy()
    if (~fin).any():  # O = 0 on rows that see no key
        if o_rows.ndim == 4:  # [B, S, H, D] vs LSE [B, H, S]
            empty = np.transpose(~fin, (0, 2, 1))
        else:                 # [total, H, D] vs LSE [H, total]
            empty = np.transpose(~fin, (1, 0))
        assert (o_rows[empty] == 0).all()


CASES = [
    # B, Hq, Hk, Sq, Sk, D, dtype, causal, window, softcap
    (1, 2, 2, 128, 128, 64, "fp16", False, None, 0.0),
    (2, 4, 2, 200, 200, 128, "bf16", True, None, 0.0),
    (1, 4, 1, 65, 130, 64, "bf16", False, None, 0.0),
    (1, 2, 2, 100, 37, 128, "fp16", True, None, 0.0),      # Sq > Sk causal: first rows see no key
    (2, 2, 2, 1, 1, 64, "bf16", True, None, 0.0),
    (1, 8, 2, 1000, 1000, 128, "bf16", True, None, 0.0),   # several key tiles, GQA 4:1
    (1, 2, 2, 777, 1300, 128, "bf16", False, None, 0.0),   # ragged both sides, Sq < Sk
    (1, 4, 4, 640, 333, 64, "fp16", True, None, 0.0),      # causal Sq > Sk over several tiles
    (1, 4, 2, 700, 700, 128, "bf16", True, (200, -1), 0.0),  # sliding window
    (1, 2, 2, 500, 500, 128, "bf16", False, (100, 37), 0.0),  # two-sided band
    (1, 2, 1, 300, 500, 64, "bf16", False, (0, 0), 0.0),      # the aligned diagonal only
    (1, 4, 2, 600, 600, 128, "bf16", True, None, 5.0),        # logit cap
    (1, 2, 2, 400, 400, 128, "fp16", False, (64, 64), 3.0),   # cap with a band
    (1, 4, 2, 300, 300, 96, "bf16", True, None, 0.0),         # D = 96 tiles
    (1, 4, 2, 600, 600, 96, "bf16", True, (200, -1), 4.0),    # D = 96, window and cap
    (2, 2, 2, 257, 257, 80, "fp16", False, None, 0.0),        # padded to the D = 96 tiles
    (1, 4, 2, 520, 520, 192, "bf16", True, None, 0.0),        # D = 192 tiles
    (1, 2, 2, 300, 300, 160, "fp16", False, (64, 64), 3.0),   # padded to D = 192, band + cap
    (1, 2, 2, 257, 257, 32, "fp16", False, None, 0.0),        # padded head dim (D = 64 kernel)
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_forward_matches_oracle(case):
    b, hq, hk, sq, sk, d, dt, causal, window, cap = case
    w = synth.small("fwdc", b, hq, hk, sq, sk, d, dt, causal, 300 + sq + sk + d)
    x = synth.make_inputs(w)
    o, lse = ab.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=causal, window=window,
                         softcap=cap)
    ab.check_device_status()
    o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, causal, window=window,
                                             softcap=cap)
    _check(o, lse, o_ref, lse_ref, str(case))


def test_forward_rescales_on_every_tile():
    """Logits that grow along the keys by about 11.5 (log2 units) per 128-key
    tile, so every tile raises each row's maximum past the 2^8 margin and the
    output accumulated so far must be rescaled: checks that path against the
    oracle (non-causal and causal)."""
    d, s = 64, 1024
    q = torch.ones(1, s, 2, d)
    j = torch.arange(s, dtype=torch.float32) / 128.0
    k = j.view(1, s, 1, 1).expand(1, s, 2, d).clone()
    g = torch.Generator().manual_seed(5)
    k += 0.05 * torch.randn(k.shape, generator=g)
    v = torch.randn(1, s, 2, d, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for causal in (False, True):
        o, lse = ab.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
        ab.check_device_status()
        o_ref, lse_ref = attn_oracle.mha_forward(q, k, v, d ** -0.5, causal)
        _check(o, lse, o_ref, lse_ref, f"rescale causal={causal}")


def test_forward_varlen_and_seqused():
    lens = [5, 130, 0, 64, 1, 257, 600]
    w = synth.Workload("fvl", 0, 4, 2, 0, 0, 128, "bf16", True, 41, n_seqs=len(lens), len_lo=0,
                       len_hi=600)
    x = synth.make_inputs(w, lengths=lens)
    cu = x.cu_seqlens_q.cuda()
    o, lse = ab.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, cu_seqlens_q=cu,
                         cu_seqlens_k=cu, max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    ab.check_device_status()
    o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, True, x.cu_seqlens_q,
                                             x.cu_seqlens_k)
    _check(o, lse, o_ref, lse_ref, "varlen")


@pytest.mark.parametrize("name", ["gqa_b2_hq32_hk8_s8192_d128_bf16_causal",
                                  "mha_b2_h16_s4096_d128_bf16"])
def test_forward_full_size_whole_heads(name):
    """The benchmark workloads' forward at full size: every row of O and LSE of
    two whole query heads against the fp64 oracle."""
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    o, lse = ab.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=w.causal)
    ab.check_device_status()
    grp = w.h_q // w.h_k
    for b, h in ((0, 0), (w.batch - 1, w.h_q - 1)):
        o_ref, lse_ref, _ = attn_oracle.head_forward(
            x.q[b, :, h].double().numpy(), x.k[b, :, h // grp].double().numpy(),
            x.v[b, :, h // grp].double().numpy(), w.scale, w.causal)
        assert_close(f"{name} O b={b} h={h}", o[b, :, h], o_ref)
        np.testing.assert_allclose(lse[b, h].cpu().double().numpy(), lse_ref, rtol=0, atol=2e-3)
