"""The input recipe of the benchmark workloads, restated independently.

The workloads give a distribution and a seed, not a generator or a draw order;
the reading taken is: one CPU generator seeded with the workload's seed, fp32
standard normals drawn in the order Q, K, V, dO (K and V with the key/value
heads), dO scaled in fp32 where the workload scales it, the cast to the dtype
last; for packed workloads the sequence lengths, uniform on the stated closed
range, come first from the same generator.
"""
import torch

from attention_backward_bwd_gb300 import synth


def test_padded_recipe():
    w = synth.WORKLOADS["mha_b4_h16_s1024_d64_fp16_causal"]
    x = synth.make_inputs(w)
    g = torch.Generator("cpu").manual_seed(1)
    q = torch.randn(4, 1024, 16, 64, generator=g)
    k = torch.randn(4, 1024, 16, 64, generator=g)
    v = torch.randn(4, 1024, 16, 64, generator=g)
    do = torch.randn(4, 1024, 16, 64, generator=g) * 0.1
    for got, want in ((x.q, q), (x.k, k), (x.v, v), (x.do, do)):
        assert got.dtype == torch.float16 and torch.equal(got, want.to(torch.float16))
    assert x.cu_seqlens_q is None


def test_gqa_recipe_heads():
    w = synth.small("recipe", 1, 8, 2, 40, 24, 16, "bf16", True, 9)
    x = synth.make_inputs(w)
    g = torch.Generator("cpu").manual_seed(9)
    q = torch.randn(1, 40, 8, 16, generator=g)
    k = torch.randn(1, 24, 2, 16, generator=g)
    assert torch.equal(x.q, q.to(torch.bfloat16)) and torch.equal(x.k, k.to(torch.bfloat16))


def test_varlen_recipe_lengths_first():
    w = synth.WORKLOADS["varlen16_h16_d128_bf16_causal"]
    g = torch.Generator("cpu").manual_seed(4)
    lengths = [int(n) for n in torch.randint(128, 8193, (16,), generator=g)]
    assert all(128 <= n <= 8192 for n in lengths)
    total = sum(lengths)
    q_head = torch.randn(total, 16, 128, generator=g)[:3]
    x = synth.make_inputs(w)
    assert x.lengths == lengths and x.lengths_k == lengths
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    assert x.cu_seqlens_q.tolist() == cu and x.cu_seqlens_q.dtype == torch.int32
    assert torch.equal(x.cu_seqlens_k, x.cu_seqlens_q)
    assert x.q.shape == (total, 16, 128)
    assert torch.equal(x.q[:3], q_head.to(torch.bfloat16))
