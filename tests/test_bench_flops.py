"""The bench's FLOP counts (no GPU needed): the closed form for unmasked and
causal problems, and the exact allowed-pair count behind windowed ones,
checked against a brute-force count over every (query, key) pair; and the
slice of the workload that the reference arm times."""
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


@pytest.mark.parametrize("causal,window,cap", [(True, None, 0.0), (False, None, 0.0),
                                               (True, (9, -1), 0.0), (False, (5, 3), 2.0)])
def test_reference_slice_is_an_exact_subproblem(causal, window, cap):
    """The reference arm times the oracle on a query head's last n rows alone
    (Sq = n against all L keys).  With bottom-right aligned masks that slice
    sees exactly the keys those rows see in the whole head, so its O, LSE, P,
    dS and dQ equal the whole head's last n rows, and its dK, dV are those
    rows' share of the whole head's sums over query rows."""
    import numpy as np
    from oracle import attn_oracle
    rng = np.random.default_rng(7)
    L, n, d = 48, 13, 16
    scale = d ** -0.5
    q, k, v, do = (rng.standard_normal((L, d)) for _ in range(4))
    full = attn_oracle.head_backward(q, k, v, do, scale, causal, window, cap)
    part = attn_oracle.head_backward(q[L - n:], k, v, do[L - n:], scale, causal, window, cap)
    for key in ("O", "LSE", "P", "dS", "dQ"):
        np.testing.assert_allclose(part[key], full[key][L - n:], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["dV"], full["P"][L - n:].T @ do[L - n:], rtol=1e-10,
                               atol=1e-12)
    np.testing.assert_allclose(part["dK"], scale * full["dS"][L - n:].T @ q[L - n:],
                               rtol=1e-10, atol=1e-12)


def test_reference_slice_flops():
    """FLOPs of a slice: 10 D per allowed pair; the whole causal head keeps the
    GPU line's 2.5 x 4 L^2 D / 2 convention."""
    w = synth.small("slice", 1, 4, 2, 64, 64, 16, "bf16", True, 3)
    x = synth.make_inputs(w)
    _, f_part, L, n = bench.oracle_sample(w, x, 10)
    assert (L, n) == (64, 10)
    assert f_part == 10.0 * 16 * sum(64 - 10 + i + 1 for i in range(10))
    _, f_full, _, n_full = bench.oracle_sample(w, x)
    assert n_full == 64 and f_full == 2.5 * 4 * 64 * 64 * 16 / 2
