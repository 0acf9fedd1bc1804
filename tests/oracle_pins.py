"""Checks that pin the fp64 oracle to facts outside itself.

Each ``pin_*`` takes the oracle module (the real one, or a copy with a planted
mistake) and raises ``AssertionError`` when the fact does not hold.  The facts:

* central finite differences of L = sum(O * dO) (dO held fixed) agree with the
  analytic dQ, dK, dV (covers MHA, GQA, causal, Sq != Sk, varlen packing);
* rowsum(P * dP) == rowsum(O * dO)  (exact algebra: sum_j P_ij dO_i.V_j = dO_i.O_i);
* all V rows equal  =>  dP constant along keys  =>  dS = 0  =>  dQ = dK = 0;
* causal, Sq == Sk: row 0 sees only key 0, so P_00 = 1, O_0 = V_0, dQ_0 = 0;
* causal, Sq < Sk: bottom-right alignment, the last query sees every key and
  the first sees keys 0 .. Sk - Sq (the window (left, 0) of the CK wrapper);
* Q = 0  =>  uniform softmax over the allowed keys (closed-form O and dV);
* Sk = 1  =>  P = 1, dQ = dK = 0, dV = sum_i dO_i;
* shift of every key row by one vector leaves dQ, dK, dV unchanged
  (rows of dS sum to zero);  permuting keys permutes dK/dV rows;
* local windows: (-1, -1) is no mask, (-1, 0) is causal, a window wider than
  both lengths is no mask; (0, 0) with Sq != Sk makes query i see only key
  i + Sk - Sq (O_i = V_{i+Sk-Sq}, dQ = dK = 0, dV = dO moved to those rows);
  a brute-force forward that writes the window as a distance band agrees;
  finite differences hold under a window;
* softcap: finite differences hold with the cap, an independent torch-autograd
  run through c * tanh(s / c) agrees, and a cap far above every logit changes
  nothing measurable;
* an independent fp64 torch-autograd run of softmax(Q K^T s) V agrees to 1e-10,
  and its logsumexp gives LSE; the same run pins the row-sampled group
  backward used at full problem sizes.
"""
from __future__ import annotations

import numpy as np
import torch

RNG = np.random.default_rng(1234)


def _rand(*shape, rng=None):
    rng = RNG if rng is None else rng
    return rng.standard_normal(shape)


def _loss(o_mod, q, k, v, do, scale, causal, cu=None):
    o, _ = o_mod.mha_forward(q, k, v, scale, causal, cu, cu)
    return float((o * do).sum())


def _fd_grad(o_mod, which, q, k, v, do, scale, causal, cu=None, h=1e-6):
    arrs = {"q": q, "k": k, "v": v}
    x = arrs[which]
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        lp = _loss(o_mod, arrs["q"], arrs["k"], arrs["v"], do, scale, causal, cu)
        x[idx] = old - h
        lm = _loss(o_mod, arrs["q"], arrs["k"], arrs["v"], do, scale, causal, cu)
        x[idx] = old
        g[idx] = (lp - lm) / (2 * h)
    return g


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-3))


FD_CASES = [
    # (B, Hq, Hk, Sq, Sk, D, causal, scale)
    (1, 2, 2, 3, 3, 4, False, 0.5),
    (1, 2, 2, 5, 5, 4, True, 0.5),
    (1, 2, 1, 5, 5, 4, True, 0.7),    # GQA, 2 query heads per kv head
    (1, 2, 1, 3, 5, 4, False, 0.5),   # Sq != Sk
    (1, 2, 2, 3, 5, 4, True, 0.5),    # causal, bottom-right alignment
    (2, 2, 1, 1, 1, 4, True, 0.5),    # S = 1
]


def pin_finite_differences(o_mod):
    for (b, hq, hk, sq, sk, d, causal, scale) in FD_CASES:
        rng = np.random.default_rng(b * 1000 + sq * 10 + sk + hq * 7 + int(causal))
        q, k, v = _rand(b, sq, hq, d, rng=rng), _rand(b, sk, hk, d, rng=rng), _rand(b, sk, hk, d, rng=rng)
        do = _rand(b, sq, hq, d, rng=rng)
        r = o_mod.mha_backward(q, k, v, do, scale, causal)
        for name, key in (("q", "dQ"), ("k", "dK"), ("v", "dV")):
            g = _fd_grad(o_mod, name, q, k, v, do, scale, causal)
            err = _rel(r[key], g)
            assert err < 1e-6, f"finite differences {key} case {(b, hq, hk, sq, sk, d, causal)}: {err}"


def pin_finite_differences_varlen(o_mod):
    rng = np.random.default_rng(77)
    lens = [2, 4, 1]
    tot = sum(lens)
    cu = np.array([0, 2, 6, 7])
    q, k, v, do = (_rand(tot, 2, 4, rng=rng), _rand(tot, 1, 4, rng=rng), _rand(tot, 1, 4, rng=rng),
                   _rand(tot, 2, 4, rng=rng))
    for causal in (False, True):
        r = o_mod.mha_backward(q, k, v, do, 0.6, causal, cu, cu)
        for name, key in (("q", "dQ"), ("k", "dK"), ("v", "dV")):
            g = _fd_grad(o_mod, name, q, k, v, do, 0.6, causal, cu)
            err = _rel(r[key], g)
            assert err < 1e-6, f"varlen finite differences {key} causal={causal}: {err}"


def _brute_forward(q, k, v, scale, off, left, right):
    """Softmax attention of one head with plain loops; key j is inside the band
    of query i when its distance d = j - i - off lies in [-left, right] (a side
    given as -1 is open)."""
    sq, sk, d = q.shape[0], k.shape[0], v.shape[1]
    o = np.zeros((sq, d))
    for i in range(sq):
        keys = [j for j in range(sk)
                if (left < 0 or j - i - off >= -left) and (right < 0 or j - i - off <= right)]
        if not keys:
            continue
        w = [np.exp(scale * float(np.dot(q[i], k[j]))) for j in keys]
        tot = sum(w)
        for wj, j in zip(w, keys):
            o[i] += (wj / tot) * v[j]
    return o


def pin_window(o_mod):
    rng = np.random.default_rng(31)
    # special cases of the window
    for sq, sk in ((4, 4), (3, 6), (6, 3)):
        q, k, v, do = _rand(sq, 5, rng=rng), _rand(sk, 5, rng=rng), _rand(sk, 5, rng=rng), \
            _rand(sq, 5, rng=rng)
        plain = o_mod.head_backward(q, k, v, do, 0.4, False)
        causal = o_mod.head_backward(q, k, v, do, 0.4, True)
        for win, ref in (((-1, -1), plain), ((sq + sk, sq + sk), plain), ((-1, 0), causal)):
            r = o_mod.head_backward(q, k, v, do, 0.4, False, win)
            for key in ("dQ", "dK", "dV", "O"):
                assert _rel(r[key], ref[key]) < 1e-14, (sq, sk, win, key)
    # window (0, 0): one key per query, at distance Sk - Sq
    sq, sk = 4, 7
    q, k, v, do = _rand(sq, 3, rng=rng), _rand(sk, 3, rng=rng), _rand(sk, 3, rng=rng), \
        _rand(sq, 3, rng=rng)
    r = o_mod.head_backward(q, k, v, do, 0.9, False, (0, 0))
    assert _rel(r["O"], v[sk - sq:]) < 1e-14
    assert np.abs(r["dQ"]).max() < 1e-13 and np.abs(r["dK"]).max() < 1e-13
    dv = np.zeros_like(v)
    dv[sk - sq:] = do
    assert _rel(r["dV"], dv) < 1e-14
    # brute force, bands of several shapes, Sq = Sk, Sq < Sk and Sq > Sk
    for sq, sk, left, right in ((6, 6, 2, 1), (4, 9, 3, 0), (9, 4, 1, -1), (5, 8, -1, 2)):
        q, k, v = _rand(sq, 4, rng=rng), _rand(sk, 4, rng=rng), _rand(sk, 4, rng=rng)
        o, _, _ = o_mod.head_forward(q, k, v, 0.5, False, (left, right))
        assert _rel(o, _brute_forward(q, k, v, 0.5, sk - sq, left, right)) < 1e-12, \
            (sq, sk, left, right)
    # causal together with a left window is the band [-left, 0]
    q, k, v = _rand(7, 4, rng=rng), _rand(9, 4, rng=rng), _rand(9, 4, rng=rng)
    o, _, _ = o_mod.head_forward(q, k, v, 0.5, True, (2, -1))
    assert _rel(o, _brute_forward(q, k, v, 0.5, 2, 2, 0)) < 1e-12


def pin_finite_differences_window(o_mod):
    rng = np.random.default_rng(55)
    for sq, sk, win, causal in ((5, 5, (1, 1), False), (3, 6, (2, 0), False), (6, 4, (1, -1), True)):
        q, k, v = _rand(1, sq, 2, 4, rng=rng), _rand(1, sk, 1, 4, rng=rng), \
            _rand(1, sk, 1, 4, rng=rng)
        do = _rand(1, sq, 2, 4, rng=rng)
        r = o_mod.mha_backward(q, k, v, do, 0.6, causal, window=win)
        arrs = {"q": q, "k": k, "v": v}
        for name, key in (("q", "dQ"), ("k", "dK"), ("v", "dV")):
            x = arrs[name]
            g = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                old = x[idx]
                x[idx] = old + 1e-6
                lp = float((o_mod.mha_forward(q, k, v, 0.6, causal, window=win)[0] * do).sum())
                x[idx] = old - 1e-6
                lm = float((o_mod.mha_forward(q, k, v, 0.6, causal, window=win)[0] * do).sum())
                x[idx] = old
                g[idx] = (lp - lm) / 2e-6
            assert _rel(r[key], g) < 1e-6, (sq, sk, win, causal, key)


def pin_softcap(o_mod):
    rng = np.random.default_rng(91)
    # torch autograd through the capped logits (shares nothing with the oracle)
    for sq, sk, causal, win, cap in ((5, 5, True, None, 1.5), (4, 7, False, (2, 1), 0.8)):
        q, k, v, do = _rand(sq, 6, rng=rng) * 2, _rand(sk, 6, rng=rng) * 2, \
            _rand(sk, 6, rng=rng), _rand(sq, 6, rng=rng)
        r = o_mod.head_backward(q, k, v, do, 0.7, causal, win, cap)
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        s = cap * torch.tanh(0.7 * (tq @ tk.T) / cap)
        i = torch.arange(sq)[:, None]
        j = torch.arange(sk)[None, :]
        band = torch.ones(sq, sk, dtype=torch.bool)
        left, right = (-1, -1) if win is None else win
        if causal:
            right = 0
        if right >= 0:
            band &= j - i - (sk - sq) <= right
        if left >= 0:
            band &= j - i - (sk - sq) >= -left
        o = torch.softmax(s.masked_fill(~band, float("-inf")), dim=1) @ tv
        (o * torch.tensor(do)).sum().backward()
        assert _rel(r["O"], o.detach().numpy()) < 1e-12
        for key, t in (("dQ", tq), ("dK", tk), ("dV", tv)):
            assert _rel(r[key], t.grad.numpy()) < 1e-10, (key, sq, sk)
    # finite differences, multi-head with GQA
    q, k, v = _rand(1, 4, 2, 4, rng=rng), _rand(1, 5, 1, 4, rng=rng), _rand(1, 5, 1, 4, rng=rng)
    do = _rand(1, 4, 2, 4, rng=rng)
    r = o_mod.mha_backward(q, k, v, do, 0.9, True, softcap=0.6)
    arrs = {"q": q, "k": k, "v": v}
    for name, key in (("q", "dQ"), ("k", "dK"), ("v", "dV")):
        x = arrs[name]
        g = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + 1e-6
            lp = float((o_mod.mha_forward(q, k, v, 0.9, True, softcap=0.6)[0] * do).sum())
            x[idx] = old - 1e-6
            lm = float((o_mod.mha_forward(q, k, v, 0.9, True, softcap=0.6)[0] * do).sum())
            x[idx] = old
            g[idx] = (lp - lm) / 2e-6
        assert _rel(r[key], g) < 1e-6, key
    # a cap far above every logit: tanh is linear there
    q, k, v, do = _rand(6, 4, rng=rng), _rand(6, 4, rng=rng), _rand(6, 4, rng=rng), \
        _rand(6, 4, rng=rng)
    a = o_mod.head_backward(q, k, v, do, 0.5, True)
    b = o_mod.head_backward(q, k, v, do, 0.5, True, None, 1e5)
    for key in ("dQ", "dK", "dV", "O"):
        assert _rel(b[key], a[key]) < 1e-8, key


def pin_delta_identity(o_mod):
    for causal in (False, True):
        q, k, v, do = _rand(7, 8), _rand(7, 8), _rand(7, 8), _rand(7, 8)
        r = o_mod.head_backward(q, k, v, do, 0.35, causal)
        d_out = o_mod.delta_from_output(r["O"], do)
        assert _rel(r["Delta"], d_out) < 1e-12, "rowsum(P*dP) != rowsum(O*dO)"
        d_direct = (r["P"] * r["dP"]).sum(axis=1)
        assert _rel(r["Delta"], d_direct) < 1e-12


def pin_equal_value_rows(o_mod):
    for causal in (False, True):
        q, k, do = _rand(6, 8), _rand(6, 8), _rand(6, 8)
        v = np.tile(_rand(1, 8), (6, 1))
        r = o_mod.head_backward(q, k, v, do, 0.4, causal)
        assert np.abs(r["dQ"]).max() < 1e-12, "equal V rows must give dQ = 0"
        assert np.abs(r["dK"]).max() < 1e-12, "equal V rows must give dK = 0"
        np.testing.assert_allclose(r["dV"], r["P"].T @ do, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["O"], v, rtol=1e-12, atol=1e-12)


def pin_causal_row0(o_mod):
    q, k, v, do = _rand(5, 4), _rand(5, 4), _rand(5, 4), _rand(5, 4)
    r = o_mod.head_backward(q, k, v, do, 0.5, True)
    assert abs(r["P"][0, 0] - 1.0) < 1e-14 and np.abs(r["P"][0, 1:]).max() == 0.0
    np.testing.assert_allclose(r["O"][0], v[0], rtol=0, atol=1e-14)
    assert np.abs(r["dQ"][0]).max() < 1e-14
    assert abs(r["LSE"][0] - 0.5 * float(q[0] @ k[0])) < 1e-12
    # upper triangle is masked
    assert np.abs(np.triu(r["P"], 1)).max() == 0.0


def pin_causal_bottom_right(o_mod):
    sq, sk = 3, 5
    q, k, v, do = _rand(sq, 4), _rand(sk, 4), _rand(sk, 4), _rand(sq, 4)
    r = o_mod.head_backward(q, k, v, do, 0.5, True)
    p = r["P"]
    assert (p[0, :3] > 0).all() and (p[0, 3:] == 0).all(), "row 0 must see keys 0..Sk-Sq"
    assert (p[2] > 0).all(), "the last query row must see every key"
    # non-causal sees everything
    r2 = o_mod.head_backward(q, k, v, do, 0.5, False)
    assert (r2["P"] > 0).all()


def pin_zero_query(o_mod):
    for causal in (False, True):
        n = 6
        q = np.zeros((n, 4))
        k, v, do = _rand(n, 4), _rand(n, 4), _rand(n, 4)
        r = o_mod.head_backward(q, k, v, do, 0.9, causal)
        cnt = np.array([i + 1 if causal else n for i in range(n)], dtype=float)
        w = np.array([[1.0 / cnt[i] if (not causal or j <= i) else 0.0 for j in range(n)]
                      for i in range(n)])
        o_exp = np.stack([v[: (i + 1 if causal else n)].mean(axis=0) for i in range(n)])
        np.testing.assert_allclose(r["O"], o_exp, rtol=1e-13, atol=1e-13)
        dv_exp = np.zeros_like(v)
        for j in range(n):
            for i in range(n):
                dv_exp[j] += w[i, j] * do[i]
        np.testing.assert_allclose(r["dV"], dv_exp, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(r["LSE"], np.log(cnt), rtol=1e-14, atol=1e-14)


def pin_single_key(o_mod):
    q, k, v, do = _rand(4, 8), _rand(1, 8), _rand(1, 8), _rand(4, 8)
    r = o_mod.head_backward(q, k, v, do, 0.3, False)
    assert np.abs(r["dQ"]).max() < 1e-15 and np.abs(r["dK"]).max() < 1e-14
    np.testing.assert_allclose(r["dV"][0], do.sum(axis=0), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(r["O"], np.tile(v, (4, 1)), rtol=1e-14, atol=1e-14)


def pin_key_shift_and_permutation(o_mod):
    q, k, v, do = _rand(6, 8), _rand(6, 8), _rand(6, 8), _rand(6, 8)
    r = o_mod.head_backward(q, k, v, do, 0.4, False)
    c = _rand(1, 8)
    r2 = o_mod.head_backward(q, k + c, v, do, 0.4, False)
    assert _rel(r2["dQ"], r["dQ"]) < 1e-10, "dQ must not change when every key moves by c"
    assert _rel(r2["dV"], r["dV"]) < 1e-10
    assert _rel(r2["dK"], r["dK"]) < 1e-10
    perm = np.array([3, 0, 5, 1, 4, 2])
    r3 = o_mod.head_backward(q, k[perm], v[perm], do, 0.4, False)
    assert _rel(r3["dQ"], r["dQ"]) < 1e-12
    assert _rel(r3["dK"], r["dK"][perm]) < 1e-12
    assert _rel(r3["dV"], r["dV"][perm]) < 1e-12


def _torch_head(q, k, v, do, scale, causal):
    q = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    s = torch.matmul(q, k.transpose(0, 1)) * scale
    if causal:
        sq, sk = s.shape
        keep = torch.ones(sq, sk, dtype=torch.bool).tril(diagonal=sk - sq)
        s = s.masked_fill(~keep, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    o = torch.matmul(torch.softmax(s, dim=-1), v)
    o.backward(torch.tensor(do, dtype=torch.float64))
    return o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def pin_torch_autograd(o_mod):
    rng = np.random.default_rng(99)
    cases = [(2, 4, 2, 9, 9, 16, True), (1, 3, 3, 7, 11, 8, False), (1, 4, 1, 12, 12, 8, True),
             (2, 2, 2, 8, 13, 8, True)]
    for (b, hq, hk, sq, sk, d, causal) in cases:
        q, k, v = (rng.standard_normal((b, sq, hq, d)), rng.standard_normal((b, sk, hk, d)),
                   rng.standard_normal((b, sk, hk, d)))
        do = rng.standard_normal((b, sq, hq, d))
        scale = d ** -0.5
        r = o_mod.mha_backward(q, k, v, do, scale, causal)
        g = hq // hk
        dk_ref, dv_ref = np.zeros_like(k), np.zeros_like(v)
        for bb in range(b):
            for h in range(hq):
                o, lse, dq, dk, dv = _torch_head(q[bb, :, h], k[bb, :, h // g], v[bb, :, h // g],
                                                 do[bb, :, h], scale, causal)
                assert _rel(r["O"][bb, :, h], o) < 1e-10
                assert _rel(r["LSE"][bb, h], lse) < 1e-10
                assert _rel(r["dQ"][bb, :, h], dq) < 1e-10
                dk_ref[bb, :, h // g] += dk
                dv_ref[bb, :, h // g] += dv
        assert _rel(r["dK"], dk_ref) < 1e-10
        assert _rel(r["dV"], dv_ref) < 1e-10
        o2, lse2 = o_mod.mha_forward(q, k, v, scale, causal)
        assert _rel(o2, r["O"]) < 1e-12 and _rel(lse2, r["LSE"]) < 1e-12


def pin_varlen_matches_padded(o_mod):
    rng = np.random.default_rng(5)
    lens = [3, 7, 5]
    cu = np.cumsum([0] + lens)
    tot = cu[-1]
    q, k, v, do = (rng.standard_normal((tot, 4, 8)), rng.standard_normal((tot, 2, 8)),
                   rng.standard_normal((tot, 2, 8)), rng.standard_normal((tot, 4, 8)))
    r = o_mod.mha_backward(q, k, v, do, 0.3, True, cu, cu)
    for b, n in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        rb = o_mod.mha_backward(q[None, sl], k[None, sl], v[None, sl], do[None, sl], 0.3, True)
        assert _rel(r["dQ"][sl], rb["dQ"][0]) < 1e-13
        assert _rel(r["dK"][sl], rb["dK"][0]) < 1e-13
        assert _rel(r["dV"][sl], rb["dV"][0]) < 1e-13
        assert _rel(r["LSE"][:, sl], rb["LSE"][0]) < 1e-13


def pin_cross_varlen_matches_padded(o_mod):
    """Packed sequences whose query and key lengths differ (cross attention,
    including a sequence with keys but no queries and one with queries but no
    keys): each sequence's gradients equal those of the same sequence alone,
    and the query-less sequence has dK = dV = 0."""
    rng = np.random.default_rng(6)
    lq, lk = [3, 0, 5, 2], [6, 4, 2, 0]
    cq, ck = np.cumsum([0] + lq), np.cumsum([0] + lk)
    q, do = rng.standard_normal((cq[-1], 4, 8)), rng.standard_normal((cq[-1], 4, 8))
    k, v = rng.standard_normal((ck[-1], 2, 8)), rng.standard_normal((ck[-1], 2, 8))
    for causal in (False, True):
        r = o_mod.mha_backward(q, k, v, do, 0.3, causal, cq, ck)
        for b in range(len(lq)):
            qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
            if lq[b] == 0:
                assert np.abs(r["dK"][ks]).max(initial=0.0) == 0
                assert np.abs(r["dV"][ks]).max(initial=0.0) == 0
                continue
            rb = o_mod.mha_backward(q[None, qs], k[None, ks], v[None, ks], do[None, qs], 0.3,
                                    causal)
            assert _rel(r["dQ"][qs], rb["dQ"][0]) < 1e-13
            if lk[b] > 0:
                assert _rel(r["dK"][ks], rb["dK"][0]) < 1e-13
                assert _rel(r["dV"][ks], rb["dV"][0]) < 1e-13
            else:
                assert np.abs(r["dQ"][qs]).max() == 0  # no keys: dQ = 0


def pin_seqused(o_mod):
    """Used lengths inside padded and packed buffers: each sequence's gradients
    equal those of its used rows alone, the unused rows change nothing (filled
    with other values, the results stay) and get zero gradients."""
    rng = np.random.default_rng(12)
    # padded: B = 3 slabs of 7 query / 9 key rows, used (5, 0, 7) / (9, 4, 2)
    uq, uk = [5, 0, 7], [9, 4, 2]
    q, do = rng.standard_normal((3, 7, 4, 8)), rng.standard_normal((3, 7, 4, 8))
    k, v = rng.standard_normal((3, 9, 2, 8)), rng.standard_normal((3, 9, 2, 8))
    for causal in (False, True):
        r = o_mod.mha_backward(q, k, v, do, 0.4, causal, seqused_q=uq, seqused_k=uk)
        q2, k2, v2, do2 = q.copy(), k.copy(), v.copy(), do.copy()
        for b in range(3):
            q2[b, uq[b]:] = 5.0
            do2[b, uq[b]:] = -3.0
            k2[b, uk[b]:] = 7.0
            v2[b, uk[b]:] = 2.0
        r2 = o_mod.mha_backward(q2, k2, v2, do2, 0.4, causal, seqused_q=uq, seqused_k=uk)
        for key in ("dQ", "dK", "dV"):
            assert _rel(r2[key], r[key]) < 1e-14, key
        for b in range(3):
            if uq[b] == 0 or uk[b] == 0:
                continue
            rb = o_mod.mha_backward(q[b:b + 1, :uq[b]], k[b:b + 1, :uk[b]], v[b:b + 1, :uk[b]],
                                    do[b:b + 1, :uq[b]], 0.4, causal)
            assert _rel(r["dQ"][b, :uq[b]], rb["dQ"][0]) < 1e-13
            assert _rel(r["dK"][b, :uk[b]], rb["dK"][0]) < 1e-13
            assert _rel(r["dV"][b, :uk[b]], rb["dV"][0]) < 1e-13
            assert np.abs(r["dQ"][b, uq[b]:]).max(initial=0.0) == 0
            assert np.abs(r["dK"][b, uk[b]:]).max(initial=0.0) == 0
    # packed: the used rows start at each sequence's offset
    cq, ck = np.array([0, 4, 10]), np.array([0, 6, 9])
    q, do = rng.standard_normal((10, 2, 4)), rng.standard_normal((10, 2, 4))
    k, v = rng.standard_normal((9, 1, 4)), rng.standard_normal((9, 1, 4))
    r = o_mod.mha_backward(q, k, v, do, 0.5, True, cq, ck, seqused_q=[3, 6], seqused_k=[6, 2])
    rb = o_mod.mha_backward(q[None, 4:10], k[None, 6:8], v[None, 6:8], do[None, 4:10], 0.5, True)
    assert _rel(r["dQ"][4:10], rb["dQ"][0]) < 1e-13 and _rel(r["dK"][6:8], rb["dK"][0]) < 1e-13
    rb = o_mod.mha_backward(q[None, 0:3], k[None, 0:6], v[None, 0:6], do[None, 0:3], 0.5, True)
    assert _rel(r["dV"][0:6], rb["dV"][0]) < 1e-13 and np.abs(r["dQ"][3]).max() == 0


def pin_empty_cases(o_mod):
    # seqlen_q == 0: dK = dV = 0
    q, do = np.zeros((1, 0, 2, 4)), np.zeros((1, 0, 2, 4))
    k, v = _rand(1, 3, 2, 4), _rand(1, 3, 2, 4)
    r = o_mod.mha_backward(q, k, v, do, 0.5, False)
    assert np.abs(r["dK"]).max() == 0 and np.abs(r["dV"]).max() == 0
    # causal, Sq > Sk: the first rows see no key -> O = 0, dQ = 0, LSE = +inf
    q, k, v, do = _rand(5, 4), _rand(2, 4), _rand(2, 4), _rand(5, 4)
    r = o_mod.head_backward(q, k, v, do, 0.5, True)
    assert np.isinf(r["LSE"][:3]).all() and np.isfinite(r["LSE"][3:]).all()
    assert np.abs(r["O"][:3]).max() == 0 and np.abs(r["dQ"][:3]).max() == 0


def pin_sympy_exact(o_mod):
    """Symbolic differentiation (sympy) of sum(O * dO) on a tiny head, evaluated
    to 30 digits: an exact gradient that shares nothing with the oracle."""
    import pytest
    sp = pytest.importorskip("sympy")
    for (sq, sk, causal) in ((2, 3, False), (2, 3, True), (3, 3, True)):
        d = 2
        rng = np.random.default_rng(sq * 10 + sk + int(causal))
        qv, kv, vv, dov = (rng.integers(-3, 4, (sq, d)) / 2, rng.integers(-3, 4, (sk, d)) / 2,
                           rng.integers(-3, 4, (sk, d)) / 2, rng.integers(-3, 4, (sq, d)) / 2)
        Q = sp.Matrix(sq, d, lambda i, j: sp.Symbol(f"q{i}_{j}"))
        K = sp.Matrix(sk, d, lambda i, j: sp.Symbol(f"k{i}_{j}"))
        V = sp.Matrix(sk, d, lambda i, j: sp.Symbol(f"v{i}_{j}"))
        scale = sp.Rational(3, 5)
        L = 0
        for i in range(sq):
            keys = [j for j in range(sk) if (not causal) or j <= i + (sk - sq)]
            w = [sp.exp(scale * sum(Q[i, t] * K[j, t] for t in range(d))) for j in keys]
            z = sum(w)
            for t in range(d):
                o_it = sum(w[a] * V[j, t] for a, j in enumerate(keys)) / z
                L += o_it * sp.Rational(str(dov[i, t]))
        subs = {}
        for M, val in ((Q, qv), (K, kv), (V, vv)):
            for i in range(M.rows):
                for j in range(M.cols):
                    subs[M[i, j]] = sp.Rational(str(val[i, j]))
        r = o_mod.head_backward(qv, kv, vv, dov, 0.6, causal)
        for M, key in ((Q, "dQ"), (K, "dK"), (V, "dV")):
            exact = np.array([[float(sp.N(sp.diff(L, M[i, j]).subs(subs), 30))
                               for j in range(M.cols)] for i in range(M.rows)])
            assert _rel(r[key], exact) < 1e-12, f"sympy {key} sq={sq} sk={sk} causal={causal}"


def pin_group_rows_autograd(o_mod):
    """The row-sampled group backward (used at full problem sizes) against an
    independent fp64 torch-autograd run, with a query-row block smaller than
    the sequence so the block loop and the causal offsets inside it are used."""
    rng = np.random.default_rng(77)
    for (b, hq, hk, sq, sk, d, causal, blk) in ((2, 4, 2, 11, 11, 8, True, 4),
                                                (1, 3, 1, 9, 13, 8, True, 5),
                                                (1, 2, 2, 7, 6, 4, False, 3)):
        q, k, v = (rng.standard_normal((b, sq, hq, d)), rng.standard_normal((b, sk, hk, d)),
                   rng.standard_normal((b, sk, hk, d)))
        do = rng.standard_normal((b, sq, hq, d))
        scale = 0.7 * d ** -0.5
        grp = hq // hk
        for bb in range(b):
            for g in range(hk):
                q_rows = [0, sq // 2, sq - 1]
                k_rows = [0, sk // 3, sk - 1]
                dq, dk, dv = o_mod.group_backward_rows(q, k, v, do, bb, g, q_rows, k_rows,
                                                       scale, causal, block=blk)
                dk_ref, dv_ref = np.zeros((sk, d)), np.zeros((sk, d))
                for hh in range(grp):
                    h = g * grp + hh
                    _, _, dq_t, dk_t, dv_t = _torch_head(q[bb, :, h], k[bb, :, g], v[bb, :, g],
                                                         do[bb, :, h], scale, causal)
                    assert _rel(dq[hh], dq_t[q_rows]) < 1e-10
                    dk_ref += dk_t
                    dv_ref += dv_t
                assert _rel(dk, dk_ref[k_rows]) < 1e-10
                assert _rel(dv, dv_ref[k_rows]) < 1e-10
    # under a window, against the full backward (pinned under windows by pin_window)
    b, hq, hk, sq, sk, d = 1, 4, 2, 13, 10, 8
    q, k, v = (rng.standard_normal((b, sq, hq, d)), rng.standard_normal((b, sk, hk, d)),
               rng.standard_normal((b, sk, hk, d)))
    do = rng.standard_normal((b, sq, hq, d))
    for win, causal, cap in (((3, 1), False, 0.0), ((2, -1), True, 0.0), (None, True, 0.4)):
        full = o_mod.mha_backward(q, k, v, do, 0.3, causal, window=win, softcap=cap)
        q_rows, k_rows = [0, 5, sq - 1], [0, 4, sk - 1]
        for g in range(hk):
            dq, dk, dv = o_mod.group_backward_rows(q, k, v, do, 0, g, q_rows, k_rows, 0.3, causal,
                                                   block=4, window=win, softcap=cap)
            for hh in range(hq // hk):
                assert _rel(dq[hh], full["dQ"][0, q_rows, g * (hq // hk) + hh]) < 1e-12
            assert _rel(dk, full["dK"][0, k_rows, g]) < 1e-12
            assert _rel(dv, full["dV"][0, k_rows, g]) < 1e-12


ALL_PINS = [pin_sympy_exact, pin_finite_differences, pin_finite_differences_varlen, pin_delta_identity,
            pin_equal_value_rows, pin_causal_row0, pin_causal_bottom_right, pin_zero_query,
            pin_single_key, pin_key_shift_and_permutation, pin_torch_autograd,
            pin_varlen_matches_padded, pin_cross_varlen_matches_padded, pin_empty_cases,
            pin_group_rows_autograd, pin_window, pin_finite_differences_window, pin_softcap,
            pin_seqused]
