"""GPU parity for grouped-query and multi-query attention (key/value heads
shared by equal consecutive groups of query heads) through fa_bwd_gqa and
fa_fwd_stats_gqa, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity import Prepared, check_case, to_np

pytestmark = pytest.mark.gpu


def gqa(name, b, h, hkv, d, s1, s2, causal, seed, **kw):
    return si.fixed(name, b, h, d, s1, s2, causal, seed, heads_kv=hkv, **kw)


SMALL = [
    gqa("gqa_g2_d128_tail", 2, 4, 2, 128, 300, 333, False, 61),
    gqa("gqa_g4_d64_causal_tail", 1, 8, 2, 64, 333, 333, True, 62),
    gqa("mqa_d128_causal", 2, 6, 1, 128, 257, 257, True, 63),
    gqa("gqa_g8_d128_s1024", 1, 16, 2, 128, 1024, 1024, False, 64),
    gqa("gqa_g2_d128_causal_s2_gt_s1", 1, 4, 2, 128, 130, 400, True, 65),
    si.Case("gqa_varlen_nan_padding_d64", 6, 64, [100, 0, 513, 3], [190, 5, 513, 0], False, 66,
            pad_q=7, pad_kv=9, heads_kv=3),
    si.Case("mqa_varlen_causal_d128", 4, 128, [129, 700, 1], [129, 700, 1], True, 67, pad_q=3, pad_kv=3,
            heads_kv=1),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c.name)
def test_gqa_parity_full(case):
    check_case(Prepared(case))


@pytest.mark.parametrize("case", SMALL[:3], ids=lambda c: c.name)
def test_gqa_forward_statistics(case):
    """O, m, l of fa_fwd_stats_gqa against the oracle forward."""
    import attention_backward_sm_gb300 as fab
    prep = Prepared(case)
    o, m, l = fab.forward_stats(prep.q, prep.k, prep.v, prep.cu_q, prep.cu_kv, case.cu_q, case.cu_kv,
                                case.causal, prep.scale)
    torch.cuda.synchronize()
    n = int(case.cu_q[-1])
    ref_o = prep.o_cpu.double().numpy()[:n]
    assert np.abs(to_np(o)[:n] - ref_o).max() <= 2e-2 * np.abs(ref_o).max()
    assert np.allclose(to_np(m)[:n], prep.m_cpu.double().numpy()[:n], rtol=1e-5, atol=1e-5)
    assert np.allclose(to_np(l)[:n], prep.l_cpu.double().numpy()[:n], rtol=1e-4, atol=1e-5)


def test_gqa_one_group_equals_multi_head():
    """heads_kv = heads through fa_bwd_gqa is the multi-head path: the same
    bits as fa_bwd in deterministic mode."""
    import attention_backward_sm_gb300 as fab
    case = si.fixed("mha_via_gqa", 2, 3, 128, 300, 300, True, 68)
    prep = Prepared(case)
    a = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    work = fab.Workspace(prep.q, case.cu_q, case.cu_kv, case.causal, fab.FA_DQ_DETERMINISTIC)
    dk = torch.empty_like(prep.k)
    dv = torch.empty_like(prep.v)
    fab.fa_bwd_preprocess(prep.o, prep.do, work.D, work.dq_acc)
    fab.fa_bwd(prep.q, prep.k, prep.v, prep.do, prep.m, prep.l, work.D, work.dq_acc, dk, dv, prep.cu_q, prep.cu_kv,
               case.cu_q, case.cu_kv, case.causal, prep.scale, fab.FA_DQ_DETERMINISTIC, work.ws)
    dq = torch.empty_like(prep.q)
    fab.fa_bwd_dq_finalize(work.dq_acc, dq, prep.scale)
    torch.cuda.synchronize()
    for x, y in zip(a, (dq, dk, dv)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("case", [
    gqa("gqa_det_g4_d128_causal", 2, 8, 2, 128, 700, 700, True, 69),
    si.Case("gqa_det_g2_d64_varlen", 4, 64, [300, 1, 513], [257, 700, 129], False, 70, pad_q=5, pad_kv=3,
            heads_kv=2),
], ids=lambda c: c.name)
def test_gqa_deterministic(case):
    import attention_backward_sm_gb300 as fab
    prep = Prepared(case)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    for a, b in zip(first, again):
        assert torch.equal(a, b)


@pytest.mark.parametrize("case,groups", [
    (gqa("gqa_b2_h32_hkv8_s4096_d128_causal", 2, 32, 8, 128, 4096, 4096, True, 71), [(0, 3), (1, 6)]),
    (gqa("mqa_b1_h16_hkv1_s2048_d64", 1, 16, 1, 64, 2048, 2048, False, 72), [(0, 0)]),
], ids=lambda x: getattr(x, "name", "groups"))
def test_gqa_full_size_sampled(case, groups):
    """Large grouped problems: the GPU runs all heads; whole groups of query
    heads are checked against the oracle (dQ per query head, dK/dV per
    shared key/value head)."""
    G = case.heads // case.kv_heads
    subset = [(b, hk * G + i) for b, hk in groups for i in range(G)]
    check_case(Prepared(case, heads_subset=subset))
