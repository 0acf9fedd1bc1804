"""Planted mistakes in a copy of the oracle (on the CPU) must each fail a pin.

A copy of the oracle source is edited in memory (one plausible slip per case:
a dropped term, a wrong sign, a transposed operand, a wrong index), loaded as a
throw-away module, and run through the pins.  If some mutant passed every pin,
the pins would not be strong enough to trust the oracle.
"""
import importlib.util
import os
import types

import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "attn_oracle.py")

MUTANTS = {
    "drop_delta": ("ds = p * (dp - delta[:, None])", "ds = p * dp"),
    "delta_sign": ("ds = p * (dp - delta[:, None])", "ds = p * (dp + delta[:, None])"),
    "dq_no_scale": ("dq = scale * (ds @ k)", "dq = ds @ k"),
    "dk_transposed": ("dk = scale * (ds.T @ q)", "dk = scale * (ds @ q[: ds.shape[1]])"),
    "dv_untransposed": ("dv = p.T @ do", "dv = p @ do"),
    "dp_wrong_operand": ("dp = do @ v.T", "dp = do @ k.T"),
    "delta_axis": ("delta = (p * dp).sum(axis=1)", "delta = (p * dp).mean(axis=1)"),
    "causal_direction": ("ok &= j <= i + (sk - sq) + right", "ok &= j >= i + (sk - sq) + right"),
    "causal_top_left": ("ok &= j <= i + (sk - sq) + right", "ok &= j <= i + right"),
    "window_left_sign": ("ok &= j >= i + (sk - sq) - left", "ok &= j >= i + (sk - sq) + left"),
    "window_left_top_left": ("ok &= j >= i + (sk - sq) - left", "ok &= j >= i - left"),
    "window_left_strict": ("ok &= j >= i + (sk - sq) - left", "ok &= j > i + (sk - sq) - left"),
    "lse_log2": ("m + np.log(np.where(any_key, ell, 1.0))", "m + np.log2(np.where(any_key, ell, 1.0))"),
    "gqa_head_map_fwd": ("_take(k, ks, h // g), _take(v, ks, h // g)", "_take(k, ks, h % hk), _take(v, ks, h % hk)"),
    "gqa_no_group_sum": ("_put(dk, ks, hkv, r[\"dK\"], add=True)", "_put(dk, ks, hkv, r[\"dK\"])"),
    "delta_from_output_axis": ("np.asarray(do, dtype=np.float64)).sum(axis=-1)", "np.asarray(do, dtype=np.float64)).sum(axis=0)"),
    "softmax_no_max_shift_sign": ("np.exp(s - m[:, None])", "np.exp(s + m[:, None])"),
    "varlen_keys_by_query_offsets": ("yield b, (slice(cq[b], cq[b] + nq),), (slice(ck[b], ck[b] + nk),)",
                                     "yield b, (slice(cq[b], cq[b] + nq),), (slice(cq[b], cq[b] + nk),)"),
    "softcap_no_derivative": ("ds = ds * (1.0 - np.tanh(scale * (q @ k.T) / softcap) ** 2)",
                              "ds = ds * 1.0"),
    "softcap_derivative_unscaled": ("ds = ds * (1.0 - np.tanh(scale * (q @ k.T) / softcap) ** 2)",
                                    "ds = ds * (1.0 - np.tanh((q @ k.T) / softcap) ** 2)"),
    "softcap_inside_scale": ("s = softcap * np.tanh(s / softcap)", "s = np.tanh(s / softcap)"),
    "seqused_ignored_padded": ("qs = slice(None) if uq is None else slice(0, uq[b])",
                               "qs = slice(None)"),
    "seqused_packed_from_zero": ("yield b, (slice(cq[b], cq[b] + nq),), (slice(ck[b], ck[b] + nk),)",
                                 "yield b, (slice(cq[b], cq[b] + nq),), (slice(0, nk),)"),
    "rows_softcap_no_derivative": ("                ds = ds * (1.0 - np.tanh(s_raw / softcap) ** 2)",
                                   "                ds = ds * 1.0"),
    # the row-sampled group backward
    "rows_drop_delta": ("            ds = p * (dp - delta[:, None])", "            ds = p * dp"),
    "rows_dv_from_ds": ("dv += p[:, k_rows].T @ doh[i0:i1]", "dv += ds[:, k_rows].T @ doh[i0:i1]"),
    "rows_window_dropped": ("allowed = allowed_pairs(ii, jj, sq, sk, causal, window)",
                            "allowed = allowed_pairs(ii, jj, sq, sk, causal)"),
    "rows_unnormalised": ("p = np.where(allowed, np.exp(s - lse[:, None]), 0.0)",
                          "p = np.where(allowed, np.exp(s - m[:, None]), 0.0)"),
}


def _load_mutant(name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found in the oracle source"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new, 1), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # a planted slip may divide by zero
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError or a shape error from the slip
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant {name} passed every pin"
