"""GPU parity for the mask variants through fa_bwd_ex / fa_fwd_stats_ex:
bottom-right causal alignment and the causal sliding window (JAX
fused_attention_stablehlo.py, sliding_window_length), against the fp64
oracle, including rows that see no key and keys no query sees."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity import Prepared, check_case, to_np

pytestmark = pytest.mark.gpu


def case(name, b, h, d, s1, s2, seed, window=0, br=False, **kw):
    return si.fixed(name, b, h, d, s1, s2, True, seed, window=window, bottom_right=br, **kw)


SMALL = [
    case("br_s1_lt_s2_d128", 1, 2, 128, 300, 700, 81, br=True),
    case("br_s1_gt_s2_d64", 1, 2, 64, 700, 300, 82, br=True),          # 400 queries see no key
    si.Case("br_varlen_nan_padding_d128", 3, 128, [100, 3, 513, 256, 0], [300, 3, 200, 256, 40], True, 83,
            pad_q=5, pad_kv=7, bottom_right=True),
    case("win256_d128", 1, 3, 128, 1000, 1000, 84, window=256),
    case("win128_d128_tail", 2, 2, 128, 517, 517, 86, window=128),
    case("win200_br_cross_d64", 1, 2, 64, 300, 900, 87, window=200, br=True),
    case("win333_s1_gt_s2_d128", 1, 2, 128, 900, 400, 88, window=333),  # top-left: late queries see nothing
    case("win300_gqa_d128", 1, 4, 128, 777, 777, 89, window=300, heads_kv=2),
    si.Case("win_br_varlen_d64", 4, 64, [129, 1, 700, 64], [300, 5, 700, 1], True, 90, window=97,
            bottom_right=True, pad_q=3, pad_kv=2),
]


@pytest.mark.parametrize("c", SMALL, ids=lambda c: c.name)
def test_mask_parity_full(c):
    check_case(Prepared(c))


@pytest.mark.parametrize("c", [SMALL[1], SMALL[3], SMALL[5], SMALL[6]], ids=lambda c: c.name)
def test_mask_forward_statistics(c):
    """O, m, l of fa_fwd_stats_ex against the oracle forward (m = -inf and
    l = 0 exactly for rows that see no key)."""
    import attention_backward_sm_gb300 as fab
    prep = Prepared(c)
    o, m, l = fab.forward_stats(prep.q, prep.k, prep.v, prep.cu_q, prep.cu_kv, c.cu_q, c.cu_kv, c.causal,
                                prep.scale, window=c.window, bottom_right=c.bottom_right)
    torch.cuda.synchronize()
    n = int(c.cu_q[-1])
    ref_o = prep.o_cpu.double().numpy()[:n]
    ref_m = prep.m_cpu.double().numpy()[:n]
    ref_l = prep.l_cpu.double().numpy()[:n]
    assert np.abs(to_np(o)[:n] - ref_o).max() <= 2e-2 * np.abs(ref_o).max()
    empty = ref_l == 0
    assert np.all(to_np(l)[:n][empty] == 0) and np.all(np.isneginf(to_np(m)[:n][empty]))
    assert np.allclose(to_np(m)[:n][~empty], ref_m[~empty], rtol=1e-5, atol=1e-5)
    assert np.allclose(to_np(l)[:n][~empty], ref_l[~empty], rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("c", [
    case("det_win333_d128", 2, 2, 128, 1500, 1500, 91, window=333),
    case("det_br_d128", 1, 3, 128, 500, 1300, 92, br=True),
    case("det_win_br_d64", 1, 2, 64, 1200, 700, 93, window=450, br=True),
], ids=lambda c: c.name)
def test_mask_deterministic(c):
    """Deterministic dQ under every mask: parity, and bitwise repeats (the
    ticket order follows the band of visited key blocks)."""
    import attention_backward_sm_gb300 as fab
    prep = Prepared(c)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    for a, b in zip(first, again):
        assert torch.equal(a, b)


def test_window_at_least_both_lengths_is_causal():
    """A window as long as both sequences together excludes nothing: the
    same bits as the plain causal mask (deterministic mode)."""
    import attention_backward_sm_gb300 as fab
    base = si.fixed("causal_ref", 1, 2, 128, 700, 700, 94, True)
    prep = Prepared(base)
    a = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    b = fab.backward(prep.q, prep.k, prep.v, prep.o, prep.do, prep.m, prep.l, prep.cu_q, prep.cu_kv, base.cu_q,
                     base.cu_kv, True, prep.scale, fab.FA_DQ_DETERMINISTIC, window=1400)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("c,n", [
    (case("win1024_b2_h16_s8192_d128", 2, 16, 128, 8192, 8192, 95, window=1024), 2),
    (case("br_b2_h16_s2048_s8192_d128", 2, 16, 128, 2048, 8192, 96, br=True), 2),
], ids=lambda x: getattr(x, "name", str(x)))
def test_mask_full_size_sampled(c, n):
    rng = np.random.default_rng(c.seed)
    units = [(b, h) for b in range(c.batch) for h in range(c.heads)]
    subset = [units[i] for i in sorted(rng.choice(len(units), size=n, replace=False))]
    check_case(Prepared(c, heads_subset=subset))


@pytest.mark.parametrize("d", [64, 128])
def test_window_one_degenerate(d):
    """W = 1 on a square problem: P = I, so dV = dO exactly in value and
    dS_ii = dP_ii - D_i = dO_i . V_i - O_i . dO_i vanishes by cancellation
    (O_i = V_i).  dQ and dK are then rounding noise and relative errors are
    undefined: they must stay within the rounding of two fp32 dot products
    of d terms (2^-14 * sum_k |O_ik dO_ik| as the bound, as for s2 = 1)."""
    c = case(f"win1_d{d}", 1, 2, d, 300, 300, 85 + d, window=1)
    prep = Prepared(c)
    dq, dk, dv = prep.run()
    ref = prep.reference()
    from parity import compare
    compare("dv", to_np(dv), ref[2])
    o = prep.o_cpu.double().numpy()
    do = prep.cpu[3].double().numpy()
    q = prep.cpu[0].double().numpy()
    k = prep.cpu[1].double().numpy()
    noise = 2.0 ** -14 * c.softmax_scale * np.abs(o * do).sum(axis=-1)[:, :, None]   # [s, H, 1]
    assert np.all(np.abs(to_np(dq)) <= noise * np.abs(k) + 1e-30)
    assert np.all(np.abs(to_np(dk)) <= noise * np.abs(q) + 1e-30)
