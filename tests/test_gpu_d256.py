"""GPU parity for head_dim 256 (the JAX cuDNN wrapper's largest flash
head dim): the tensor-core forward with 64-row key blocks, and the
backward that splits the head dimension over two CTAs per key block,
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity import Prepared, check_case, compare, to_np

pytestmark = pytest.mark.gpu


def c256(name, b, h, s1, s2, causal, seed, **kw):
    return si.fixed(name, b, h, 256, s1, s2, causal, seed, **kw)


SMALL = [
    c256("d256_noncausal_tail", 2, 2, 300, 333, False, 301),
    c256("d256_causal_tail", 1, 3, 517, 517, True, 302),
    c256("d256_causal_s2_gt_s1", 1, 2, 130, 400, True, 303),
    si.Case("d256_varlen_nan_padding", 3, 256, [1, 257, 64, 0, 100], [190, 257, 65, 5, 0], False, 304,
            pad_q=7, pad_kv=9),
    c256("d256_gqa_window_br", 1, 4, 700, 900, True, 305, heads_kv=2, window=300, bottom_right=True),
    c256("d256_mqa_causal", 2, 3, 129, 129, True, 306, heads_kv=1),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c.name)
def test_d256_backward_parity(case):
    check_case(Prepared(case))


@pytest.mark.parametrize("case", SMALL[:2] + SMALL[3:5], ids=lambda c: c.name)
def test_d256_forward_parity(case):
    import attention_backward_sm_gb300 as fab
    q, k, v, _ = case.tensors()
    dev = torch.device("cuda")
    cu_q, cu_kv = torch.from_numpy(case.cu_q).to(dev), torch.from_numpy(case.cu_kv).to(dev)
    o, m, l = fab.forward_stats(q.to(dev), k.to(dev), v.to(dev), cu_q, cu_kv, case.cu_q, case.cu_kv, case.causal,
                                case.softmax_scale, window=case.window, bottom_right=case.bottom_right)
    torch.cuda.synchronize()
    o64, m64, l64 = oracle.forward_packed(q, k, v, case.cu_q, case.cu_kv, case.softmax_scale, case.causal,
                                          window=case.window, bottom_right=case.bottom_right)
    n = int(case.cu_q[-1])
    o, m, l = to_np(o)[:n], to_np(m)[:n], to_np(l)[:n]
    empty = l64[:n] == 0
    compare("O", o, o64[:n], np.broadcast_to(empty[:, :, None], o.shape))
    assert np.all(l[empty] == 0) and np.all(np.isneginf(m[empty]))
    np.testing.assert_allclose(m[~empty], m64[:n][~empty], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(l[~empty], l64[:n][~empty], rtol=1e-4)


@pytest.mark.parametrize("case", [SMALL[1], SMALL[3], SMALL[4]], ids=lambda c: c.name)
def test_d256_deterministic(case):
    import attention_backward_sm_gb300 as fab
    prep = Prepared(case)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    for a, b in zip(first, again):
        assert torch.equal(a, b)


def test_d256_lse_backward():
    import attention_backward_sm_gb300 as fab
    case = c256("d256_lse", 1, 2, 400, 400, True, 307)
    prep = Prepared(case)
    lse_cpu = torch.from_numpy(oracle.lse_from_stats(prep.m_cpu, prep.l_cpu)).to(torch.float32)
    out = fab.backward_lse(prep.q, prep.k, prep.v, prep.o, prep.do, lse_cpu.cuda(), prep.cu_q, prep.cu_kv,
                           case.cu_q, case.cu_kv, True, prep.scale)
    torch.cuda.synchronize()
    q, k, v, do = prep.cpu
    ref = oracle.backward_packed_lse(q, k, v, prep.o_cpu, do, lse_cpu, case.cu_q, case.cu_kv, prep.scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), out, ref[:3]):
        compare(name, to_np(g), r)


@pytest.mark.parametrize("case", [c256("d256_b2_h8_s4096_causal", 2, 8, 4096, 4096, True, 308),
                                  c256("d256_b1_h8_s4096_noncausal", 1, 8, 4096, 4096, False, 309)],
                         ids=lambda c: c.name)
def test_d256_full_size_sampled(case):
    rng = np.random.default_rng(case.seed)
    units = [(b, h) for b in range(case.batch) for h in range(case.heads)]
    subset = [units[i] for i in sorted(rng.choice(len(units), size=2, replace=False))]
    check_case(Prepared(case, heads_subset=subset))
