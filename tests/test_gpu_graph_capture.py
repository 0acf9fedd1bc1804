"""attn_bwd captured in a CUDA graph and replayed.

A launch-bound caller (small heads, short sequences) removes the host cost of
the three launches by capturing them once and replaying the graph.  The
capture must record exactly the work of an eager call: replays give the eager
results bit for bit (deterministic mode), and read whatever the captured input
buffers hold at replay time.
"""
import pytest
import torch

import attention_backward_bwd_gb300 as ab
from attention_backward_bwd_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs(varlen, seed, d=128):
    if varlen:
        w = synth.Workload("graph_varlen", 0, 4, 2, 0, 0, d, "bf16", True, seed, n_seqs=4,
                           len_lo=1, len_hi=600)
        return w, synth.make_inputs(w, lengths=[200, 0, 513, 128])
    w = synth.small("graph", 2, 8, 2, 600, 600, d, "bf16", True, seed)
    return w, synth.make_inputs(w)


@pytest.mark.parametrize("varlen,d", [(False, 128), (True, 128), (False, 192), (True, 256)],
                         ids=["padded", "varlen", "padded-d192", "varlen-d256"])
def test_attn_bwd_replays_in_a_cuda_graph(varlen, d):
    w, x = _inputs(varlen, 21, d)
    _, x2 = _inputs(varlen, 22, d)
    dev = "cuda"
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    kw = dict(causal=w.causal, deterministic=True)
    if varlen:
        mx = max(x.lengths)
        kw.update(cu_seqlens_q=x.cu_seqlens_q.to(dev), cu_seqlens_k=x.cu_seqlens_k.to(dev),
                  max_seqlen_q=mx, max_seqlen_k=mx)
    fwd_kw = {k_: v_ for k_, v_ in kw.items() if k_ != "deterministic"}
    o, lse = ab.attn_fwd(q, k, v, **fwd_kw)
    ws = ab.alloc_workspace(q, kw.get("cu_seqlens_q"), True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    args = (q, k, v, o, lse, do)
    outs = dict(workspace=ws, dq=dq, dk=dk, dv=dv)

    # eager call first (one-time per-device setup must not happen inside a capture)
    ab.attn_bwd(*args, **kw, **outs)
    ab.check_device_status()
    ref = [t.clone() for t in (dq, dk, dv)]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ab.attn_bwd(*args, **kw, **outs)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ab.attn_bwd(*args, **kw, **outs)

    for _ in range(2):
        for t in (dq, dk, dv):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ab.check_device_status()
        for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.equal(got, r), f"replay {name} differs from the eager call"

    # new values in the captured input buffers: the replay reads them
    q2, k2, v2, do2 = (t.to(dev) for t in (x2.q, x2.k, x2.v, x2.do))
    o2, lse2 = ab.attn_fwd(q2, k2, v2, **fwd_kw)
    eager2 = ab.attn_bwd(q2, k2, v2, o2, lse2, do2, **kw)
    for dst, src in zip(args, (q2, k2, v2, o2, lse2, do2)):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    ab.check_device_status()
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), eager2):
        assert torch.equal(got, r), f"replay on new inputs: {name} differs"
