"""GPU tests of the individual kernels through the C ABI: tensor-core tile
forms, the bounded-wait error path, the preprocess, the forward and the
postprocess."""
import numpy as np
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth
from oracle import attn_oracle
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_diag_mma_tile(mode, d, dtype):
    g = torch.Generator("cpu").manual_seed(100 + mode * 10 + d)
    ka = d if mode == 0 else 128
    a = torch.randn(128, ka, generator=g).to(DT[dtype])
    b = torch.randn(128, d, generator=g).to(DT[dtype])
    c = ab.diag_mma(mode, a.cuda(), b.cuda())
    ab.check_device_status()
    a64, b64 = a.double(), b.double()
    if mode == 0:
        ref = a64 @ b64.T
    elif mode == 1:
        ref = a64 @ b64
    else:
        ref = a64.T @ b64
    err = (c.cpu().double() - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), f"mode {mode}: max err {err}"


def test_diag_tanh_accuracy():
    """The logit cap's tanh (1 - 2 / (e^{2x} + 1) from the hardware exponential
    and reciprocal): absolute error <= 2e-6 against float64 over the range the
    cap feeds it, exact limits at +-inf-like inputs, odd to within the bound."""
    x = torch.cat([torch.linspace(-40.0, 40.0, 1 << 20),
                   torch.tensor([0.0, 1e-6, -1e-6, 1e4, -1e4, 89.0, -89.0])])
    y = ab.diag_tanh(x.cuda()).cpu().double()
    ref = torch.tanh(x.double())
    assert (y - ref).abs().max().item() <= 2e-6
    assert y[-4].item() == 1.0 and y[-3].item() == -1.0
    assert (y + ab.diag_tanh(-x.cuda()).cpu().double()).abs().max().item() <= 4e-6


def test_device_wait_timeout_is_reported():
    ab.diag_wait_timeout(50_000_000)  # 50 ms on a barrier nothing completes
    with pytest.raises(ab.AttnError) as e:
        ab.check_device_status()
    assert e.value.code == -8
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
    ab.check_device_status()


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64)])
def test_preprocess_delta_and_lse2(dtype, d):
    w = synth.small("pre", 2, 4, 2, 300, 300, d, dtype, False, 21)
    x = synth.make_inputs(w)
    o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, False)
    o = torch.tensor(o_ref).to(DT[dtype])
    lse = torch.tensor(lse_ref, dtype=torch.float32)
    dev = [t.cuda() for t in (x.q, x.k, x.v, x.do)]
    ws = ab.alloc_workspace(dev[0])
    ab.attn_bwd(*dev[:3], o.cuda(), lse.cuda(), dev[3], workspace=ws, stage="pre")
    ab.check_device_status()
    offs, rows = ab.workspace_layout(2, 300, 4, d)
    wsc = ws.cpu()
    delta = wsc[offs["delta"]:offs["delta"] + 4 * rows * 4].view(torch.float32).view(4, rows)
    lse2 = wsc[offs["lse2"]:offs["lse2"] + 4 * rows * 4].view(torch.float32).view(4, rows)
    sr = 384  # 300 rounded up to the 128-row tile
    want = attn_oracle.delta_from_output(o.double().numpy(), x.do.double().numpy())  # [B,S,H]
    for b in range(2):
        got = delta[:, b * sr: b * sr + 300].double().numpy().T  # [S, H]
        np.testing.assert_allclose(got, want[b], rtol=1e-4, atol=1e-4)
        assert (delta[:, b * sr + 300:(b + 1) * sr] == 0).all()
        got2 = lse2[:, b * sr: b * sr + 300].double().numpy()
        np.testing.assert_allclose(got2, lse_ref[b] * np.log2(np.e), rtol=1e-6, atol=1e-5)
    dqacc = wsc[offs["dqaccum"]:offs["dqaccum"] + 4 * rows * d * 4].view(torch.float32)
    assert (dqacc == 0).all()


FWD_CASES = [
    (1, 2, 2, 128, 128, 64, "fp16", False),
    (2, 4, 2, 200, 200, 128, "bf16", True),
    (1, 4, 1, 65, 130, 64, "bf16", False),
    (1, 2, 2, 100, 37, 128, "fp16", True),   # Sq > Sk causal: first rows see no key
    (2, 2, 2, 1, 1, 64, "bf16", True),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=str)
def test_forward_matches_oracle(case):
    b, hq, hk, sq, sk, d, dtype, causal = case
    w = synth.small("fwd", b, hq, hk, sq, sk, d, dtype, causal, 31)
    x = synth.make_inputs(w)
    o, lse = ab.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=causal)
    ab.check_device_status()
    o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, causal)
    assert_close("O", o, o_ref)
    lc = lse.cpu().double().numpy()
    fin = np.isfinite(lse_ref)
    assert (np.isinf(lc) == ~fin).all()
    np.testing.assert_allclose(lc[fin], lse_ref[fin], rtol=0, atol=2e-3)


def test_forward_varlen():
    lens = [5, 130, 64, 1, 257]
    w = synth.Workload("fvl", 0, 4, 2, 0, 0, 128, "bf16", True, 41, n_seqs=5, len_lo=1, len_hi=300)
    x = synth.make_inputs(w, lengths=lens)
    cu = x.cu_seqlens_q.cuda()
    o, lse = ab.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, cu_seqlens_q=cu,
                         cu_seqlens_k=cu, max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    ab.check_device_status()
    o_ref, lse_ref = attn_oracle.mha_forward(x.q, x.k, x.v, w.scale, True, x.cu_seqlens_q,
                                             x.cu_seqlens_k)
    assert_close("O", o, o_ref)
    np.testing.assert_allclose(lse.cpu().double().numpy(), lse_ref, rtol=0, atol=2e-3)
