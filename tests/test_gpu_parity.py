"""GPU parity: libfabwd.so (through the C ABI) against the fp64 oracle.

Small and medium cases compare every element; the full-size workloads of
the target specification compare every element of a sample of
(sequence, head) units that the oracle computes one by one (the GPU still
runs the whole problem in the launch configuration the benchmark uses).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity import Prepared, check_case, to_np

pytestmark = pytest.mark.gpu


def fixed(name, b, h, d, s1, s2, causal, seed, **kw):
    return si.fixed(name, b, h, d, s1, s2, causal, seed, **kw)


SMALL = [
    si.cfg1(),
    si.cfg2(),
    fixed("d64_tail_noncausal", 2, 3, 64, 200, 333, False, 12),
    fixed("d64_tail_causal", 2, 3, 64, 333, 333, True, 13),
    fixed("d128_tail_causal", 1, 4, 128, 300, 300, True, 14),
    fixed("d128_causal_s2_gt_s1", 1, 2, 128, 130, 400, True, 15),     # keys no query sees
    fixed("d128_causal_s2_lt_s1", 1, 2, 128, 400, 130, True, 16),
    fixed("d64_short_129", 1, 2, 64, 129, 129, True, 17),
    si.Case("varlen_nan_padding_d128", 3, 128, [1, 257, 128, 0, 64], [190, 257, 128, 5, 0], False, 18,
            pad_q=7, pad_kv=9),
    si.Case("varlen_nan_padding_d64_causal", 4, 64, [100, 3, 513, 256], [100, 3, 513, 256], True, 19,
            pad_q=13, pad_kv=13),
    # shapes of the SK-16 article's test matrix with head_dim in {64, 128} (tests/golden/sk16_test_shapes.txt)
    fixed("sk16_01_b8_h8_s320_d64", 8, 8, 64, 320, 320, False, 21),
    fixed("sk16_05_b8_h8_s32_d64", 8, 8, 64, 32, 32, False, 25),
    fixed("sk16_06_b8_h4_s64_d128", 8, 4, 128, 64, 64, False, 26),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c.name)
def test_parity_full(case):
    prep = Prepared(case)
    check_case(prep)


def sampled(case, n, seed):
    rng = np.random.default_rng(seed)
    units = [(b, h) for b in range(case.batch) for h in range(case.heads)
             if case.q_lens[b] > 0 and case.kv_lens[b] > 0]
    idx = rng.choice(len(units), size=min(n, len(units)), replace=False)
    return [units[i] for i in sorted(idx)]


FULL = [
    (si.cfg3(True), 3),
    (si.cfg3(False), 2),
    (si.cfg4(), 3),
    (si.cfg5(), 3),
    (fixed("sk16_02_b8_h8_s2432_d64", 8, 8, 64, 2432, 2432, False, 22), 2),
]


@pytest.mark.parametrize("case,n", FULL, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_parity_full_size_sampled(case, n):
    subset = sampled(case, n, seed=case.seed)
    # the longest sequence of a varlen batch is always among the checked units
    if case.batch > 1:
        bmax = int(np.argmax(case.q_lens))
        if all(b != bmax for b, _ in subset):
            subset = subset + [(bmax, 0)]
    prep = Prepared(case, heads_subset=subset)
    check_case(prep)


def test_dv_column_sum_all_heads_cfg2():
    """sum_j dV_j = sum_i dO_i holds for every head at any size (rows of P
    sum to one); checked on all heads with the library's own forward."""
    import attention_backward_sm_gb300 as fab
    case = si.cfg2()
    q, k, v, do = (t.cuda() for t in case.tensors())
    cu_q = torch.from_numpy(case.cu_q).cuda()
    cu_kv = torch.from_numpy(case.cu_kv).cuda()
    o, m, l = fab.forward_stats(q, k, v, cu_q, cu_kv, case.cu_q, case.cu_kv, False, case.softmax_scale)
    dq, dk, dv = fab.backward(q, k, v, o, do, m, l, cu_q, cu_kv, case.cu_q, case.cu_kv, False, case.softmax_scale)
    torch.cuda.synchronize()
    for b in range(case.batch):
        rq = slice(int(case.cu_q[b]), int(case.cu_q[b + 1]))
        rk = slice(int(case.cu_kv[b]), int(case.cu_kv[b + 1]))
        lhs = to_np(dv[rk]).sum(axis=0)
        rhs = to_np(do[rq]).sum(axis=0)
        assert np.linalg.norm(lhs - rhs) <= 1e-2 * np.linalg.norm(rhs)
        # sum_j dK_j = 0 (rowsum of dS is zero): small against the size of dK
        dkb = to_np(dk[rk])
        assert np.linalg.norm(dkb.sum(axis=0)) <= 1e-2 * np.linalg.norm(dkb)


@pytest.mark.parametrize("d", [64, 128])
def test_single_key_degenerate(d):
    """s2 = 1: P = 1, so dP_i0 = dO_i . V_0 = D_i and dS = 0 exactly; dQ and
    dK vanish by cancellation and relative errors are undefined.  dV must
    match (sum of dO); dQ and dK must stay within the rounding of the two fp32
    dot products that cancel: |dS_i0| <= 2 * 2^-17 * sum_k |O_ik dO_ik| for a
    128-term fp32 sum (2^-14 used as the bound factor for headroom)."""
    case = fixed(f"single_key_d{d}", 1, 2, d, 77, 1, False, 11 + d)
    prep = Prepared(case)
    dq, dk, dv = prep.run()
    ref = prep.reference()
    from parity import compare
    compare("dv", to_np(dv), ref[2])
    o = prep.o_cpu.double().numpy()
    do = prep.cpu[3].double().numpy()
    q = prep.cpu[0].double().numpy()
    k = prep.cpu[1].double().numpy()
    noise = np.abs(o * do).sum(axis=-1)                       # [s1, H]
    bound_q = 2.0 ** -14 * case.softmax_scale * noise[:, :, None] * np.abs(k[0])[None, :, :]
    bound_k = 2.0 ** -14 * case.softmax_scale * (noise[:, :, None] * np.abs(q)).sum(axis=0)
    assert np.all(np.abs(to_np(dq)) <= bound_q + 1e-30)
    assert np.all(np.abs(to_np(dk)[0]) <= bound_k + 1e-30)


@pytest.mark.parametrize("case", [
    si.fixed("det_d128_causal_tail", 2, 3, 128, 700, 700, True, 51),
    si.Case("det_d64_varlen_cross", 3, 64, [300, 1, 513], [257, 700, 129], False, 52, pad_q=5, pad_kv=3),
    si.fixed("det_d128_noncausal_square_tail", 2, 3, 128, 700, 700, False, 53),
    si.fixed("det_d64_noncausal_square", 1, 2, 64, 1024, 1024, False, 54, heads_kv=1),
], ids=lambda c: c.name)
def test_deterministic_mode(case):
    """FA_DQ_DETERMINISTIC: parity with the oracle, and dQ bitwise identical
    across runs (every dQ row is summed by one CTA in a fixed key-block
    order).  dK and dV come from the same key-block sweep as in the atomic
    mode, so they carry the same bits there."""
    import attention_backward_sm_gb300 as fab
    prep = Prepared(case)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    for _ in range(2):
        again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    anyorder = prep.run(dq_mode=fab.FA_DQ_ATOMIC)
    assert torch.equal(first[1], anyorder[1]) and torch.equal(first[2], anyorder[2])


def test_deterministic_full_size_cfg3_causal_bitwise():
    """Full-size causal batch in deterministic mode: two runs agree bit for bit
    and the sampled heads match the oracle."""
    import attention_backward_sm_gb300 as fab
    case = si.cfg3(True)
    subset = sampled(case, 2, seed=7)
    prep = Prepared(case, heads_subset=subset)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    assert torch.equal(first[0], again[0])


def test_deterministic_full_size_noncausal_bitwise():
    """Full-size batch without a mask in deterministic mode: two runs agree
    bit for bit and the sampled heads match the oracle."""
    import attention_backward_sm_gb300 as fab
    case = si.cfg3(False)
    subset = sampled(case, 2, seed=8)
    prep = Prepared(case, heads_subset=subset)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    assert torch.equal(first[0], again[0])


def test_deterministic_full_size_cross_bitwise():
    """Cross attention with unequal query and key block counts per sequence
    (cfg5's lengths): two deterministic runs agree bit for bit and sampled
    heads match the oracle."""
    import attention_backward_sm_gb300 as fab
    case = si.cfg5()
    subset = sampled(case, 2, seed=9)
    prep = Prepared(case, heads_subset=subset)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    for a, b in zip(first, again):
        assert torch.equal(a, b)


def test_deterministic_unit_larger_than_the_ring_bound():
    """160 key blocks per (sequence, head), more than the GPU holds CTAs at
    once (no CTA of the deterministic mode waits on another, so the unit
    size is free).  Properties that hold at any size: bitwise repeats,
    agreement with the any-order mode up to fp32 summation order, and
    sum_j dV_j = sum_i dO_i."""
    import attention_backward_sm_gb300 as fab
    case = si.fixed("det_ring_d64_s20480", 1, 2, 64, 20480, 20480, False, 55)
    q, k, v, do = (t.cuda() for t in case.tensors())
    cu = torch.from_numpy(case.cu_q).cuda()
    o, m, l = fab.forward_stats(q, k, v, cu, cu, case.cu_q, case.cu_kv, False, case.softmax_scale)
    run = lambda mode: fab.backward(q, k, v, o, do, m, l, cu, cu, case.cu_q, case.cu_kv, False,
                                    case.softmax_scale, mode)
    first = run(fab.FA_DQ_DETERMINISTIC)
    again = run(fab.FA_DQ_DETERMINISTIC)
    anyorder = run(fab.FA_DQ_ATOMIC)
    torch.cuda.synchronize()
    fab.fa_check_device_status()
    for a, b, c in zip(first, again, anyorder):
        assert torch.equal(a, b)
        a64, c64 = to_np(a), to_np(c)
        assert np.linalg.norm(a64 - c64) <= 1e-3 * np.linalg.norm(c64)
    dv = to_np(first[2])
    rhs = to_np(do).sum(axis=0)
    assert np.linalg.norm(dv.sum(axis=0) - rhs) <= 1e-2 * np.linalg.norm(rhs)


# Causal grids whose key blocks have sweeps of very different lengths launch
# heavy-first in chunks of (sequence, key/value head) units: 32 MiB of
# query-side data (Q, dO in bf16 and fp32 dQ per query head) per chunk.
# These shapes leave a short last chunk; the checked heads include its units.
CHUNKED = [
    # 8 MiB per unit -> chunks of 4 units: {4, 1}
    (fixed("chunk_d128_b1_h5_s8192_causal", 1, 5, 128, 8192, 8192, True, 31), [(0, 0), (0, 3), (0, 4)]),
    # d = 64, 16384 rows: 8 MiB per unit -> {4, 1}
    (fixed("chunk_d64_b1_h5_s16384_causal", 1, 5, 64, 16384, 16384, True, 32), [(0, 1), (0, 4)]),
    # grouped (2 query heads per key/value head), 16 MiB per unit -> {2, 1}
    (fixed("chunk_gqa_b1_h6_hkv3_s16384_causal", 1, 6, 128, 16384, 16384, True, 33, heads_kv=3),
     [(0, 4), (0, 5)]),
    # head_dim 256 (64-row query blocks), 16 MiB per unit -> {2, 1}
    (fixed("chunk_d256_b1_h3_s8192_causal", 1, 3, 256, 8192, 8192, True, 34), [(0, 0), (0, 2)]),
    # bottom-right diagonal with s2 slightly above s1: sweeps still uneven; 6 units, one chunk
    (fixed("chunk_br_b2_h3_s4096_4608", 2, 3, 128, 4096, 4608, True, 35, bottom_right=True), [(0, 2), (1, 0)]),
]


@pytest.mark.parametrize("case,subset", CHUNKED, ids=lambda x: getattr(x, "name", "units"))
def test_chunked_launch_order_sampled(case, subset):
    check_case(Prepared(case, heads_subset=subset))
