"""Seeded synthetic inputs for the attention backward workloads.

This module only draws random numbers and names workload shapes. It holds none
of the attention arithmetic, so both the fp64 oracle (tests) and the CUDA path
(tests, bench) can take their inputs from it without sharing any of the method.

Draw order (one ``torch.Generator('cpu')`` per case, fp32 draws, cast last):
varlen lengths (if any), then Q, K, V, dO.  K and V carry the key/value heads
(``h_k``).  ``do_scale`` multiplies dO in fp32 before the cast.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-backward problem shape.

    For varlen workloads ``n_seqs`` sequences with lengths uniform in
    ``[len_lo, len_hi]`` are packed into ``[total, H, D]`` and ``batch``/``seqlen``
    are ignored.
    """

    name: str
    batch: int
    h_q: int
    h_k: int
    seqlen_q: int
    seqlen_k: int
    head_dim: int
    dtype: str
    causal: bool
    seed: int
    do_scale: float = 1.0
    deterministic: bool = False
    n_seqs: int = 0
    len_lo: int = 0
    len_hi: int = 0
    window: tuple = (-1, -1)  # local mask (left, right), -1 = unbounded side
    softcap: float = 0.0      # logit cap c (0 = none)

    @property
    def windowed(self) -> bool:
        return tuple(self.window) != (-1, -1)

    @property
    def varlen(self) -> bool:
        return self.n_seqs > 0

    @property
    def scale(self) -> float:
        return self.head_dim ** -0.5


# The five problem shapes the attention-backward benchmark is quoted on, and extensions
# of them (deterministic, window, logit cap, head dims above 128).
WORKLOADS = {
    "mha_b1_h2_s128_d64_fp16": Workload(
        "mha_b1_h2_s128_d64_fp16", 1, 2, 2, 128, 128, 64, "fp16", False, 0),
    "mha_b4_h16_s1024_d64_fp16_causal": Workload(
        "mha_b4_h16_s1024_d64_fp16_causal", 4, 16, 16, 1024, 1024, 64, "fp16", True, 1,
        do_scale=0.1),
    "mha_b2_h16_s4096_d128_bf16": Workload(
        "mha_b2_h16_s4096_d128_bf16", 2, 16, 16, 4096, 4096, 128, "bf16", False, 2),
    "mha_b2_h16_s4096_d128_bf16_causal": Workload(
        "mha_b2_h16_s4096_d128_bf16_causal", 2, 16, 16, 4096, 4096, 128, "bf16", True, 2),
    "gqa_b2_hq32_hk8_s8192_d128_bf16_causal": Workload(
        "gqa_b2_hq32_hk8_s8192_d128_bf16_causal", 2, 32, 8, 8192, 8192, 128, "bf16", True, 3),
    "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_det": Workload(
        "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_det", 2, 32, 8, 8192, 8192, 128, "bf16", True,
        3, deterministic=True),
    "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_win1024": Workload(
        "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_win1024", 2, 32, 8, 8192, 8192, 128, "bf16", True,
        3, window=(1024, -1)),
    "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_cap30": Workload(
        "gqa_b2_hq32_hk8_s8192_d128_bf16_causal_cap30", 2, 32, 8, 8192, 8192, 128, "bf16", True,
        3, softcap=30.0),
    # other head dimensions, same shape as the MHA S=4096 workload: 96 (its own kernel),
    # above 128 (the wide kernels)
    "mha_b2_h16_s4096_d96_bf16_causal": Workload(
        "mha_b2_h16_s4096_d96_bf16_causal", 2, 16, 16, 4096, 4096, 96, "bf16", True, 2),
    "mha_b2_h16_s4096_d256_bf16_causal": Workload(
        "mha_b2_h16_s4096_d256_bf16_causal", 2, 16, 16, 4096, 4096, 256, "bf16", True, 2),
    "mha_b2_h16_s4096_d192_bf16_causal": Workload(
        "mha_b2_h16_s4096_d192_bf16_causal", 2, 16, 16, 4096, 4096, 192, "bf16", True, 2),
    "varlen16_h16_d128_bf16_causal": Workload(
        "varlen16_h16_d128_bf16_causal", 0, 16, 16, 0, 0, 128, "bf16", True, 4,
        n_seqs=16, len_lo=128, len_hi=8192),
}


@dataclasses.dataclass
class Inputs:
    """fp16/bf16 CPU tensors in [B, S, H, D] (or packed [total, H, D] for varlen)."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    cu_seqlens_q: Optional[torch.Tensor] = None  # int32 [n_seqs + 1]
    cu_seqlens_k: Optional[torch.Tensor] = None
    lengths: Optional[list] = None      # query lengths (varlen)
    lengths_k: Optional[list] = None    # key lengths (varlen)


def draw_lengths(g: torch.Generator, n: int, lo: int, hi: int) -> list:
    """Sequence lengths uniform in [lo, hi] (both ends included)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(w: Workload, lengths: Optional[list] = None,
                lengths_k: Optional[list] = None) -> Inputs:
    """Draw the inputs of workload ``w`` from its seed (N(0,1) entries).

    Varlen: ``lengths`` are the query lengths (drawn if not given) and
    ``lengths_k`` the key lengths (default: the same, self-attention)."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    dt = DTYPES[w.dtype]
    if w.varlen:
        if lengths is None:
            lengths = draw_lengths(g, w.n_seqs, w.len_lo, w.len_hi)
        if lengths_k is None:
            lengths_k = lengths
        assert len(lengths_k) == len(lengths)
        qs = (int(sum(lengths)), w.h_q, w.head_dim)
        ks = (int(sum(lengths_k)), w.h_k, w.head_dim)
        cu = cu_from_lengths(lengths)
        cu_k = cu_from_lengths(lengths_k)
    else:
        qs = (w.batch, w.seqlen_q, w.h_q, w.head_dim)
        ks = (w.batch, w.seqlen_k, w.h_k, w.head_dim)
        cu = cu_k = None
    q = torch.randn(qs, generator=g)
    k = torch.randn(ks, generator=g)
    v = torch.randn(ks, generator=g)
    do = torch.randn(qs, generator=g)
    if w.do_scale != 1.0:
        do = do * w.do_scale
    return Inputs(q.to(dt), k.to(dt), v.to(dt), do.to(dt), cu, cu_k, lengths, lengths_k)


def small(name: str, batch: int, h_q: int, h_k: int, sq: int, sk: int, d: int, dtype: str,
          causal: bool, seed: int, deterministic: bool = False) -> Workload:
    """A small ad-hoc workload for parity and edge-case tests."""
    return Workload(name, batch, h_q, h_k, sq, sk, d, dtype, causal, seed,
                    deterministic=deterministic)
