"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each test would fail for a plausible slip in the oracle: a dropped D term,
a wrong sign, a transposed operand, scale on the wrong gradient, a flipped
causal mask or an off-by-one in the packed offsets.

  * finite differences of L = sum(O * dO) through the oracle forward
    (pins dQ, dK, dV and the scale placement, for any mask);
  * a two-key example worked by hand;
  * closed forms at Q = 0 (uniform softmax, and prefix means under the
    top-left causal mask) and at s2 = 1;
  * gradient invariants: sum_j dV_j = sum_i dO_i, sum_j dK_j = 0 (from
    rowsum(dS) = 0), dQ unchanged when every key is shifted by one vector,
    D = rowsum(P * dP);
  * torch float64 autograd of a naive softmax attention (a library routine
    used only as an independent check).
"""
import math

import numpy as np
import pytest
import torch

from oracle import backward_head, backward_packed, forward_head, forward_packed, rowsum_o_do


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- finite differences
def _fd_check(s1, s2, d, scale, causal, seed, hstep=1e-6):
    q, k, v, do = rnd((s1, d), seed), rnd((s2, d), seed + 1), rnd((s2, d), seed + 2), rnd((s1, d), seed + 3)

    def loss(q_, k_, v_):
        o, _, _ = forward_head(q_, k_, v_, scale, causal)
        return float((o * do).sum())

    o, m, l = forward_head(q, k, v, scale, causal)
    dq, dk, dv, _ = backward_head(q, k, v, o, do, m, l, scale, causal)
    for name, t, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(t)
        for idx in np.ndindex(t.shape):
            tp, tm = t.copy(), t.copy()
            tp[idx] += hstep
            tm[idx] -= hstep
            args_p = {"q": (tp, k, v), "k": (q, tp, v), "v": (q, k, tp)}[name]
            args_m = {"q": (tm, k, v), "k": (q, tm, v), "v": (q, k, tm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * hstep)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7, err_msg=f"d{name}")


@pytest.mark.parametrize("s1,s2,d,scale,causal", [
    (5, 5, 3, 0.7, False),
    (5, 5, 3, 0.7, True),
    (4, 7, 2, 1 / math.sqrt(2), False),   # cross, s1 < s2
    (4, 7, 2, 1.3, True),                 # causal with keys no query sees
    (6, 3, 4, 0.5, True),                 # causal with s2 < s1
])
def test_finite_differences(s1, s2, d, scale, causal):
    _fd_check(s1, s2, d, scale, causal, seed=11 * s1 + s2 + int(causal))


def test_finite_differences_packed_varlen():
    """FD through the packed entry points: two sequences, two heads,
    different q and kv lengths; pins the offset arithmetic."""
    H, d, scale = 2, 3, 0.8
    cu_q = np.array([0, 3, 7], dtype=np.int32)
    cu_kv = np.array([0, 4, 6], dtype=np.int32)
    q, k, v = rnd((7, H, d), 1), rnd((6, H, d), 2), rnd((6, H, d), 3)
    do = rnd((7, H, d), 4)
    for causal in (False, True):
        o, m, l = forward_packed(q, k, v, cu_q, cu_kv, scale, causal)
        dq, dk, dv, _ = backward_packed(q, k, v, o, do, m, l, cu_q, cu_kv, scale, causal)

        def loss(q_, k_, v_):
            o_, _, _ = forward_packed(q_, k_, v_, cu_q, cu_kv, scale, causal)
            return float((o_ * do).sum())

        h = 1e-6
        for t, g, slot in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            num = np.zeros_like(t)
            for idx in np.ndindex(t.shape):
                tp, tm = t.copy(), t.copy()
                tp[idx] += h
                tm[idx] -= h
                ap = [q, k, v]
                am = [q, k, v]
                ap[slot], am[slot] = tp, tm
                num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7)


# ---------------------------------------------------------------- worked example
def test_two_key_example_by_hand():
    """s1 = 1, s2 = 2, d = 1, scale = 1, q = ln 3, keys (1, 0), values
    (2, -2), dO = 1.  By hand: scores (ln 3, 0) so P = (3/4, 1/4), m = ln 3,
    l = 1 + 1/3 = 4/3, O = 3/2 - 1/2 = 1.  dV = P * dO = (3/4, 1/4).
    dP = dO * v = (2, -2), D = O * dO = 1, dS = P * (dP - D) = (3/4, -3/4).
    dQ = dS . k = 3/4, dK = dS * q = (3/4 ln 3, -3/4 ln 3)."""
    q = np.array([[math.log(3.0)]])
    k = np.array([[1.0], [0.0]])
    v = np.array([[2.0], [-2.0]])
    do = np.array([[1.0]])
    o, m, l = forward_head(q, k, v, 1.0, False)
    np.testing.assert_allclose(m, [math.log(3.0)], rtol=1e-15)
    np.testing.assert_allclose(l, [4.0 / 3.0], rtol=1e-15)
    np.testing.assert_allclose(o, [[1.0]], rtol=1e-15)
    dq, dk, dv, D = backward_head(q, k, v, o, do, m, l, 1.0, False)
    np.testing.assert_allclose(D, [1.0], rtol=1e-15)
    np.testing.assert_allclose(dv, [[0.75], [0.25]], rtol=1e-15)
    np.testing.assert_allclose(dq, [[0.75]], rtol=1e-15)
    np.testing.assert_allclose(dk, [[0.75 * math.log(3.0)], [-0.75 * math.log(3.0)]], rtol=1e-14)


# ---------------------------------------------------------------- closed forms
def test_q_zero_noncausal_closed_form():
    """Q = 0: every score is 0, P = 1/s2, O_i = mean_j V_j, m = 0, l = s2;
    dV_j = mean_i... = (1/s2) sum_i dO_i, dK = 0,
    dQ_i = scale/s2 * sum_j (dO_i . (V_j - Vbar)) K_j."""
    s1, s2, d, scale = 6, 9, 5, 0.37
    q = np.zeros((s1, d))
    k, v, do = rnd((s2, d), 5), rnd((s2, d), 6), rnd((s1, d), 7)
    o, m, l = forward_head(q, k, v, scale, False)
    vbar = v.mean(axis=0)
    np.testing.assert_allclose(m, 0.0, atol=0)
    np.testing.assert_allclose(l, float(s2), rtol=1e-15)
    np.testing.assert_allclose(o, np.broadcast_to(vbar, o.shape), rtol=1e-13, atol=1e-14)
    dq, dk, dv, _ = backward_head(q, k, v, o, do, m, l, scale, False)
    np.testing.assert_allclose(dv, np.broadcast_to(do.sum(axis=0) / s2, dv.shape), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)
    want = np.zeros((s1, d))
    for i in range(s1):
        for j in range(s2):
            want[i] += scale / s2 * float(do[i] @ (v[j] - vbar)) * k[j]
    np.testing.assert_allclose(dq, want, rtol=1e-12, atol=1e-13)


def test_q_zero_causal_prefix_means():
    """Q = 0 under the top-left causal mask: query i averages keys 0..i, so
    O_i is the prefix mean of V and dV_j = sum_{i >= j} dO_i / (i + 1).
    A flipped mask (j >= i) would give suffix means instead."""
    s, d, scale = 7, 3, 0.9
    q = np.zeros((s, d))
    k, v, do = rnd((s, d), 8), rnd((s, d), 9), rnd((s, d), 10)
    o, m, l = forward_head(q, k, v, scale, True)
    for i in range(s):
        np.testing.assert_allclose(o[i], v[: i + 1].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert l[i] == pytest.approx(i + 1, rel=1e-15)
    dq, dk, dv, _ = backward_head(q, k, v, o, do, m, l, scale, True)
    for j in range(s):
        want = sum(do[i] / (i + 1) for i in range(j, s))
        np.testing.assert_allclose(dv[j], want, rtol=1e-13, atol=1e-14)
    for i in range(s):
        want = np.zeros(d)
        for j in range(i + 1):
            want += scale / (i + 1) * float(do[i] @ (v[j] - o[i])) * k[j]
        np.testing.assert_allclose(dq[i], want, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    """s2 = 1: P = 1 for every query, O = V_0, dS = 0, so dQ = dK = 0 and
    dV_0 = sum_i dO_i."""
    s1, d = 5, 4
    q, k, v, do = rnd((s1, d), 12), rnd((1, d), 13), rnd((1, d), 14), rnd((s1, d), 15)
    o, m, l = forward_head(q, k, v, 0.5, causal)
    dq, dk, dv, _ = backward_head(q, k, v, o, do, m, l, 0.5, causal)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)
    np.testing.assert_allclose(dv[0], do.sum(axis=0), rtol=1e-14)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    s1, s2, d, scale = 40, 40, 16, 0.25
    q, k, v, do = rnd((s1, d), 20), rnd((s2, d), 21), rnd((s2, d), 22), rnd((s1, d), 23)
    o, m, l = forward_head(q, k, v, scale, causal)
    dq, dk, dv, D = backward_head(q, k, v, o, do, m, l, scale, causal)
    # sum_j dV_j = sum_i dO_i (rows of P sum to 1)
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-12, atol=1e-12)
    # sum_j dK_j = scale * sum_i (sum_j dS_ij) Q_i = 0
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # shifting all keys by c adds a per-row constant to the scores: P, O are
    # unchanged and dQ changes by scale * rowsum(dS) * c = 0
    c = rnd((1, d), 24)
    o2, m2, l2 = forward_head(q, k + c, v, scale, causal)
    np.testing.assert_allclose(o2, o, rtol=1e-11, atol=1e-12)
    dq2, _, _, _ = backward_head(q, k + c, v, o2, do, m2, l2, scale, causal)
    np.testing.assert_allclose(dq2, dq, rtol=1e-10, atol=1e-11)
    # D = rowsum(P * dP) with P from torch's softmax of the masked scores
    x = torch.tensor(scale * (q @ k.T))
    if causal:
        x = x.masked_fill(torch.triu(torch.ones(s1, s2, dtype=torch.bool), 1), float("-inf"))
    p = torch.softmax(x, dim=1).numpy()
    np.testing.assert_allclose(D, (p * (do @ v.T)).sum(axis=1), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(D, rowsum_o_do(o, do), rtol=0, atol=0)


# ---------------------------------------------------------------- library check
@pytest.mark.parametrize("s1,s2,d,causal", [(9, 9, 8, False), (9, 9, 8, True), (5, 11, 6, False), (12, 4, 6, True)])
def test_against_torch_autograd(s1, s2, d, causal):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = rnd((s1, d), 30), rnd((s2, d), 31), rnd((s2, d), 32), rnd((s1, d), 33)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    x = scale * tq @ tk.T
    if causal:
        x = x.masked_fill(torch.triu(torch.ones(s1, s2, dtype=torch.bool), 1), float("-inf"))
    out = torch.softmax(x, dim=1) @ tv
    out.backward(torch.tensor(do))
    o, m, l = forward_head(q, k, v, scale, causal)
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(m + np.log(l), torch.logsumexp(x, dim=1).detach().numpy(), rtol=1e-12)
    dq, dk, dv, _ = backward_head(q, k, v, o, do, m, l, scale, causal)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- packed edge cases
def test_packed_padding_and_empty_sequences():
    """Padding rows and empty sequences give exact zeros; an empty key set
    gives dQ = 0 for its queries and m = -inf, l = 0."""
    H, d, scale = 2, 4, 0.5
    cu_q = np.array([0, 3, 3, 5], dtype=np.int32)     # sequence 1 has no queries
    cu_kv = np.array([0, 4, 6, 6], dtype=np.int32)    # sequence 2 has no keys
    q, do = rnd((7, H, d), 40), rnd((7, H, d), 41)    # two padding rows
    k, v = rnd((8, H, d), 42), rnd((8, H, d), 43)     # two padding rows
    for causal in (False, True):
        o, m, l = forward_packed(q, k, v, cu_q, cu_kv, scale, causal)
        assert np.all(o[3:5] == 0) and np.all(np.isneginf(m[3:5])) and np.all(l[3:5] == 0)
        dq, dk, dv, _ = backward_packed(q, k, v, o, do, m, l, cu_q, cu_kv, scale, causal)
        assert np.all(dq[3:] == 0)            # empty key set, then padding
        assert np.all(dk[6:] == 0) and np.all(dv[6:] == 0)   # padding keys
        # keys of sequence 1 are seen by no query: exact zeros
        assert np.all(dk[4:6] == 0) and np.all(dv[4:6] == 0)


def test_heads_subset_matches_full():
    H, d, scale = 3, 4, 0.5
    cu = np.array([0, 5, 9], dtype=np.int32)
    q, k, v, do = (rnd((9, H, d), s) for s in (50, 51, 52, 53))
    o, m, l = forward_packed(q, k, v, cu, cu, scale, True)
    full = backward_packed(q, k, v, o, do, m, l, cu, cu, scale, True)
    sub = [(1, 2), (0, 0)]
    o2, m2, l2 = forward_packed(q, k, v, cu, cu, scale, True, heads_subset=sub)
    part = backward_packed(q, k, v, o2, do, m2, l2, cu, cu, scale, True, heads_subset=sub)
    for b, h in sub:
        rows = slice(cu[b], cu[b + 1])
        for a, bb in zip(full[:3], part[:3]):
            np.testing.assert_array_equal(a[rows, h], bb[rows, h])


# ---------------------------------------------------------------- grouped-query attention
@pytest.mark.parametrize("hq,hkv,causal", [(4, 2, False), (4, 2, True), (3, 1, True)])
def test_gqa_finite_differences(hq, hkv, causal):
    """Query heads sharing a key/value head: finite differences of
    L = sum(O * dO) through the packed forward pin dK and dV of the shared
    head (sums over the group) as well as dQ."""
    d, scale = 3, 0.6
    cu_q = np.array([0, 4, 7], dtype=np.int32)
    cu_kv = np.array([0, 5, 8], dtype=np.int32)
    q, k, v = rnd((7, hq, d), 61), rnd((8, hkv, d), 62), rnd((8, hkv, d), 63)
    do = rnd((7, hq, d), 64)
    o, m, l = forward_packed(q, k, v, cu_q, cu_kv, scale, causal)
    dq, dk, dv, _ = backward_packed(q, k, v, o, do, m, l, cu_q, cu_kv, scale, causal)

    def loss(q_, k_, v_):
        o_, _, _ = forward_packed(q_, k_, v_, cu_q, cu_kv, scale, causal)
        return float((o_ * do).sum())

    h = 1e-6
    for t, g, slot in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(t)
        for idx in np.ndindex(t.shape):
            tp, tm = t.copy(), t.copy()
            tp[idx] += h
            tm[idx] -= h
            ap, am = [q, k, v], [q, k, v]
            ap[slot], am[slot] = tp, tm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7)


def test_gqa_with_one_group_is_multi_head():
    """hkv = hq reduces to the per-head definition exactly."""
    H, d, scale = 3, 4, 0.5
    cu = np.array([0, 6], dtype=np.int32)
    q, k, v, do = (rnd((6, H, d), s) for s in (70, 71, 72, 73))
    o, m, l = forward_packed(q, k, v, cu, cu, scale, True)
    dq, dk, dv, _ = backward_packed(q, k, v, o, do, m, l, cu, cu, scale, True)
    for h in range(H):
        oh, mh, lh = forward_head(q[:, h], k[:, h], v[:, h], scale, True)
        r = backward_head(q[:, h], k[:, h], v[:, h], oh, do[:, h], mh, lh, scale, True)
        np.testing.assert_array_equal(dq[:, h], r[0])
        np.testing.assert_array_equal(dk[:, h], r[1])
        np.testing.assert_array_equal(dv[:, h], r[2])
