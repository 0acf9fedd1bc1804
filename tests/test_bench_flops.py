"""The bench's FLOP counts (no GPU needed): the closed form for unmasked and
causal problems, and the exact allowed-pair count behind windowed ones,
checked against a brute-force count over every (query, key) pair."""
import itertools

import pytest

import bench
from attention_backward_bwd_gb300 import synth


def _brute_pairs(sq, sk, causal, window):
    left, right = window
    if causal:
        right = 0
    off = sk - sq
    return sum(1 for i, j in itertools.product(range(sq), range(sk))
               if (left < 0 or j >= i + off - left) and (right < 0 or j <= i + off + right))


@pytest.mark.parametrize("sq,sk,causal,window", [
    (37, 37, True, (8, -1)), (20, 50, False, (3, 5)), (50, 20, True, (-1, -1)),
    (33, 33, False, (0, 0)), (40, 17, False, (-1, 2)), (16, 64, True, (100, -1)),
])
def test_window_pairs_exact(sq, sk, causal, window):
    assert bench.window_pairs(sq, sk, causal, window) == _brute_pairs(sq, sk, causal, window)


def test_bench_flops_per_workload():
    w = synth.WORKLOADS["gqa_b2_hq32_hk8_s8192_d128_bf16_causal"]
    assert bench.bwd_flops(w) == 2.5 * 4 * 2 * 32 * 8192 * 8192 * 128 / 2
    ww = synth.WORKLOADS["gqa_b2_hq32_hk8_s8192_d128_bf16_causal_win1024"]
    pairs = 1024 * 1025 // 2 + (8192 - 1024) * 1025  # rows before / after the window fills
    assert bench.bwd_flops(ww) == 10.0 * 128 * 32 * 2 * pairs
    wc = synth.WORKLOADS["gqa_b2_hq32_hk8_s8192_d128_bf16_causal_cap30"]
    assert bench.bwd_flops(wc) == bench.bwd_flops(w)  # the cap adds no MMA work
