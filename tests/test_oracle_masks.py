"""Pins of the oracle's mask variants: bottom-right causal alignment and the
sliding window (JAX fused_attention_stablehlo.py, sliding_window_length).

  * the page's worked window example (tests/golden/sliding_window_example.txt);
  * reductions to other masks: bottom-right with s1 = s2 is top-left, a single
    bottom-right query sees every key, a window longer than both sequences is
    plain causal;
  * closed forms: W = 1 (each query sees only its own key, P = I) and Q = 0
    (O is the mean of V over the window);
  * finite differences of L = sum(O * dO) through the oracle forward, for
    rows that see no key as well, and through the packed entry points;
  * torch float64 autograd of softmax attention with the mask given as an
    explicit table.
"""
import os

import numpy as np
import pytest
import torch

from oracle import backward_head, backward_packed, forward_head, forward_packed, visible

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sliding_window_example.txt")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_window_example_from_the_page():
    lines = [ln for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    W = int(lines[0].split()[1])
    n = int(lines[1].split()[1])
    want = np.zeros((n, n), dtype=bool)
    for ln in lines[2:]:
        qi, keys = ln.split(":")
        for j in keys.split():
            want[int(qi), int(j)] = True
    assert np.array_equal(visible(n, n, True, window=W), want)
    assert np.array_equal(visible(n, n, True, window=W, bottom_right=True), want)


def test_mask_reductions():
    for s in (1, 5, 9):
        assert np.array_equal(visible(s, s, True, bottom_right=True), visible(s, s, True))
    for s2 in (1, 4, 11):
        assert visible(1, s2, True, bottom_right=True).all()          # one query: the last key is its own
        assert np.array_equal(visible(3, s2, True, window=3 + s2), visible(3, s2, True))
        assert np.array_equal(visible(3, s2, True, window=3 + s2, bottom_right=True),
                              visible(3, s2, True, bottom_right=True))
    # bottom-right with more queries than keys: the first s1 - s2 queries see nothing
    v = visible(7, 4, True, bottom_right=True)
    assert not v[:3].any() and v[3:].any(axis=1).all()
    with pytest.raises(ValueError):
        visible(3, 3, False, window=2)
    with pytest.raises(ValueError):
        visible(3, 3, False, bottom_right=True)


def test_window_one_closed_form():
    """W = 1 on a square problem: P = I, so O = V, dV = dO and dS = 0,
    hence dQ = dK = 0 exactly, and D_i = V_i . dO_i."""
    s, d = 6, 4
    q, k, v, do = rnd((s, d), 1), rnd((s, d), 2), rnd((s, d), 3), rnd((s, d), 4)
    for br in (False, True):
        o, m, l = forward_head(q, k, v, 0.9, True, window=1, bottom_right=br)
        np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
        np.testing.assert_allclose(l, 1.0, rtol=0, atol=0)
        dq, dk, dv, D = backward_head(q, k, v, o, do, m, l, 0.9, True, window=1, bottom_right=br)
        np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)
        assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
        np.testing.assert_allclose(D, (v * do).sum(axis=1), rtol=1e-14)


@pytest.mark.parametrize("s1,s2,W,br", [(9, 9, 3, False), (5, 9, 4, True), (9, 6, 2, True), (7, 4, 5, False)])
def test_q_zero_window_means(s1, s2, W, br):
    """Q = 0: every visible key has the same score, so O_i is the mean of V
    over the keys query i sees, and dV_j sums dO_i / n_i over the queries
    that see key j (n_i = size of query i's window)."""
    d = 3
    q = np.zeros((s1, d))
    k, v, do = rnd((s2, d), 5), rnd((s2, d), 6), rnd((s1, d), 7)
    off = s2 - s1 if br else 0
    o, m, l = forward_head(q, k, v, 0.7, True, window=W, bottom_right=br)
    dq, dk, dv, _ = backward_head(q, k, v, o, do, m, l, 0.7, True, window=W, bottom_right=br)
    dv_want = np.zeros_like(v)
    for i in range(s1):
        lo, hi = max(0, i + off - W + 1), min(s2, i + off + 1)   # keys lo .. hi-1
        if hi <= lo:
            assert np.all(o[i] == 0) and l[i] == 0 and m[i] == -np.inf
            continue
        np.testing.assert_allclose(o[i], v[lo:hi].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert l[i] == hi - lo
        dv_want[lo:hi] += do[i] / (hi - lo)
    np.testing.assert_allclose(dv, dv_want, rtol=1e-13, atol=1e-14)
    assert np.abs(dk).max() < 1e-13                                 # Q = 0


def _fd(s1, s2, d, scale, W, br, seed, h=1e-6):
    q, k, v, do = rnd((s1, d), seed), rnd((s2, d), seed + 1), rnd((s2, d), seed + 2), rnd((s1, d), seed + 3)

    def loss(q_, k_, v_):
        return float((forward_head(q_, k_, v_, scale, True, W, br)[0] * do).sum())

    o, m, l = forward_head(q, k, v, scale, True, W, br)
    grads = backward_head(q, k, v, o, do, m, l, scale, True, W, br)
    for which, t in enumerate((q, k, v)):
        num = np.zeros_like(t)
        for idx in np.ndindex(t.shape):
            tp, tm = t.copy(), t.copy()
            tp[idx] += h
            tm[idx] -= h
            a = [q, k, v]
            a[which] = tp
            lp = loss(*a)
            a[which] = tm
            num[idx] = (lp - loss(*a)) / (2 * h)
        np.testing.assert_allclose(grads[which], num, rtol=1e-6, atol=1e-7, err_msg="dq dk dv"[3 * which:3 * which + 2])


@pytest.mark.parametrize("s1,s2,W,br", [
    (5, 8, 0, True),     # bottom-right, more keys than queries
    (8, 5, 0, True),     # bottom-right, first three queries see nothing
    (7, 7, 3, False),    # window, top-left
    (6, 9, 2, True),     # window, bottom-right
    (9, 6, 4, False),    # window, top-left, last queries see a shrinking window
])
def test_finite_differences_masks(s1, s2, W, br):
    _fd(s1, s2, 3, 0.8, W, br, seed=s1 * 31 + s2 + W)


def test_finite_differences_packed_masks():
    """Per-sequence alignment: the bottom-right offset uses each sequence's
    own lengths."""
    H, d, scale = 2, 2, 0.6
    cu_q = np.array([0, 3, 8], dtype=np.int32)
    cu_kv = np.array([0, 6, 9], dtype=np.int32)
    q, k, v, do = rnd((8, H, d), 1), rnd((9, H, d), 2), rnd((9, H, d), 3), rnd((8, H, d), 4)
    for W in (0, 2):
        o, m, l = forward_packed(q, k, v, cu_q, cu_kv, scale, True, window=W, bottom_right=True)
        grads = backward_packed(q, k, v, o, do, m, l, cu_q, cu_kv, scale, True, window=W, bottom_right=True)
        for b in range(2):
            qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_kv[b], cu_kv[b + 1]
            for hh in range(H):
                ob, mb, lb = forward_head(q[qs:qe, hh], k[ks:ke, hh], v[ks:ke, hh], scale, True, W, True)
                np.testing.assert_array_equal(o[qs:qe, hh], ob)
        h = 1e-6
        for which, t in enumerate((q, k, v)):
            for idx in [(0, 0, 0), (2, 1, 1), (t.shape[0] - 1, 0, 1)]:
                tp, tm = t.copy(), t.copy()
                tp[idx] += h
                tm[idx] -= h
                a = [q, k, v]
                a[which] = tp
                lp = float((forward_packed(*a, cu_q, cu_kv, scale, True, window=W, bottom_right=True)[0] * do).sum())
                a[which] = tm
                lm = float((forward_packed(*a, cu_q, cu_kv, scale, True, window=W, bottom_right=True)[0] * do).sum())
                assert abs(grads[which][idx] - (lp - lm) / (2 * h)) < 1e-6


@pytest.mark.parametrize("s1,s2,W,br", [(6, 10, 3, True), (10, 6, 0, True), (8, 8, 5, False)])
def test_against_torch_autograd_masks(s1, s2, W, br):
    """torch float64 autograd with the mask written out as a table of the
    keys each query sees (rows that see nothing are dropped from the loss)."""
    d, scale = 4, 0.75
    q, k, v, do = rnd((s1, d), 9), rnd((s2, d), 10), rnd((s2, d), 11), rnd((s1, d), 12)
    off = s2 - s1 if br else 0
    table = np.zeros((s1, s2), dtype=bool)
    for i in range(s1):
        for j in range(s2):
            table[i, j] = j <= i + off and (W == 0 or j > i + off - W)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    rows = torch.tensor(table.any(axis=1))
    x = scale * tq @ tk.T
    x = x.masked_fill(~torch.tensor(table), float("-inf"))[rows]
    o = torch.softmax(x, dim=1) @ tv
    (o * torch.tensor(do)[rows]).sum().backward()
    oo, m, l = forward_head(q, k, v, scale, True, W, br)
    dq, dk, dv, _ = backward_head(q, k, v, oo, do, m, l, scale, True, W, br)
    np.testing.assert_allclose(oo[rows.numpy()], o.detach().numpy(), rtol=1e-12, atol=1e-13)
    for g, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=1e-10, atol=1e-12)
