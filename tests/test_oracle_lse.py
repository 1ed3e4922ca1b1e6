"""Pins of the oracle's single-statistic backward (lse = m + log l, the
reading of the float32 softmax_stat that JAX's cuDNN wrapper keeps per
query row)."""
import numpy as np
import pytest
import scipy.special

from oracle import (backward_head, backward_head_lse, backward_packed, backward_packed_lse, forward_head,
                    forward_packed, lse_from_stats, masked_scores)


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("causal,window,br", [(False, 0, False), (True, 0, False), (True, 3, True), (True, 0, True)])
def test_lse_is_logsumexp(causal, window, br):
    """lse_from_stats of the forward statistics equals scipy's logsumexp of
    the masked scaled scores (a library routine), -inf where a row sees no key."""
    q, k, v = rnd((9, 4), 1), rnd((6, 4), 2), rnd((6, 4), 3)
    _, m, l = forward_head(q, k, v, 0.7, causal, window, br)
    x = masked_scores(q, k, 0.7, causal, window, br)
    want = scipy.special.logsumexp(x, axis=1)
    got = lse_from_stats(m, l)
    np.testing.assert_allclose(got[np.isfinite(want)], want[np.isfinite(want)], rtol=1e-14)
    assert np.array_equal(np.isneginf(got), np.isneginf(want))


def test_lse_q_zero_closed_form():
    """Q = 0, non-causal: every scaled score is 0, so lse = log(s2)."""
    s2 = 7
    _, m, l = forward_head(np.zeros((3, 4)), rnd((s2, 4), 4), rnd((s2, 4), 5), 0.9, False)
    np.testing.assert_allclose(lse_from_stats(m, l), np.log(s2), rtol=1e-15)


@pytest.mark.parametrize("causal,window,br", [(False, 0, False), (True, 0, False), (True, 2, False), (True, 0, True)])
def test_lse_backward_matches_two_statistics_and_fd(causal, window, br):
    """The lse form gives the gradients of the (m, l) form, and both match
    finite differences of sum(O * dO) through the oracle forward."""
    s1, s2, d, scale = 6, 5, 3, 0.8
    q, k, v, do = rnd((s1, d), 6), rnd((s2, d), 7), rnd((s2, d), 8), rnd((s1, d), 9)
    o, m, l = forward_head(q, k, v, scale, causal, window, br)
    a = backward_head(q, k, v, o, do, m, l, scale, causal, window, br)
    b = backward_head_lse(q, k, v, o, do, lse_from_stats(m, l), scale, causal, window, br)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)
    h = 1e-6
    for which, t in enumerate((q, k, v)):
        num = np.zeros_like(t)
        for idx in np.ndindex(t.shape):
            tp, tm = t.copy(), t.copy()
            tp[idx] += h
            tm[idx] -= h
            args = [q, k, v]
            args[which] = tp
            lp = float((forward_head(*args, scale, causal, window, br)[0] * do).sum())
            args[which] = tm
            lm = float((forward_head(*args, scale, causal, window, br)[0] * do).sum())
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(b[which], num, rtol=1e-6, atol=1e-7)


def test_lse_packed_matches_two_statistics():
    cu_q = np.array([0, 4, 4, 9], dtype=np.int32)
    cu_kv = np.array([0, 3, 6, 11], dtype=np.int32)
    q, k, v, do = rnd((10, 4, 3), 1), rnd((12, 2, 3), 2), rnd((12, 2, 3), 3), rnd((10, 4, 3), 4)
    for causal, br in ((False, False), (True, True)):
        o, m, l = forward_packed(q, k, v, cu_q, cu_kv, 0.6, causal, bottom_right=br)
        a = backward_packed(q, k, v, o, do, m, l, cu_q, cu_kv, 0.6, causal, bottom_right=br)
        b = backward_packed_lse(q, k, v, o, do, lse_from_stats(m, l), cu_q, cu_kv, 0.6, causal, bottom_right=br)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)
