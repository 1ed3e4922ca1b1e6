"""GPU parity of the tensor-core forward statistics (fa_fwd_stats_ex:
O, m, l) against the fp64 oracle forward, on cases chosen to exercise the
online softmax: score ranges that grow from block to block (the running
maximum moves, O is rescaled), long rows, every mask, grouped heads, empty
sequences and NaN padding."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity import compare, to_np

pytestmark = pytest.mark.gpu


def run_forward(case, q, k, v):
    import attention_backward_sm_gb300 as fab
    dev = torch.device("cuda")
    cu_q, cu_kv = torch.from_numpy(case.cu_q).to(dev), torch.from_numpy(case.cu_kv).to(dev)
    o, m, l = fab.forward_stats(q.to(dev), k.to(dev), v.to(dev), cu_q, cu_kv, case.cu_q, case.cu_kv, case.causal,
                                case.softmax_scale, window=case.window, bottom_right=case.bottom_right)
    torch.cuda.synchronize()
    fab.fa_check_device_status()
    return o, m, l


def check_forward(case, q, k, v):
    o, m, l = run_forward(case, q, k, v)
    o64, m64, l64 = oracle.forward_packed(q, k, v, case.cu_q, case.cu_kv, case.softmax_scale, case.causal,
                                          window=case.window, bottom_right=case.bottom_right)
    nq = int(case.cu_q[-1])
    o, m, l = to_np(o)[:nq], to_np(m)[:nq], to_np(l)[:nq]
    empty = l64[:nq] == 0
    compare("O", o, o64[:nq], np.broadcast_to(empty[:, :, None], o.shape))
    assert np.array_equal(np.isneginf(m), np.isneginf(m64[:nq]))
    assert np.all(l[empty] == 0)
    np.testing.assert_allclose(m[~empty], m64[:nq][~empty], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(l[~empty], l64[:nq][~empty], rtol=1e-4)


CASES = [
    si.fixed("fwd_long_d128_scale1", 1, 2, 128, 2048, 2048, False, 201, scale=1.0),
    si.fixed("fwd_d64_causal_multiblock", 2, 3, 64, 700, 700, True, 202),
    si.fixed("fwd_window_br_gqa", 1, 4, 128, 900, 1300, True, 203, heads_kv=2, window=300, bottom_right=True),
    si.fixed("fwd_br_s1_gt_s2", 1, 2, 128, 600, 250, True, 204, bottom_right=True),
    si.Case("fwd_varlen_empty_nan_padding", 3, 128, [0, 130, 257, 40], [50, 0, 300, 129], False, 205,
            pad_q=6, pad_kv=5),
    si.Case("fwd_varlen_window_d64", 2, 64, [500, 1, 129], [500, 1, 129], True, 206, window=77, pad_q=2, pad_kv=2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_forward_parity(case):
    check_forward(case, *case.tensors()[:3])


@pytest.mark.parametrize("grow", [True, False], ids=["growing_scores", "shrinking_scores"])
def test_forward_running_max_moves(grow):
    """Keys whose norm grows (or shrinks) along the sequence: with growth the
    row maximum rises in almost every key block, so the lazily rescaled
    accumulator is rescaled repeatedly; without it never after the first."""
    case = si.fixed("fwd_rescale", 1, 2, 128, 256, 1536, False, 207, scale=0.5)
    q, k, v, _ = case.tensors()
    ramp = torch.linspace(0.2, 3.0, k.shape[0]) if grow else torch.linspace(3.0, 0.2, k.shape[0])
    k = (k.float() * ramp[:, None, None]).to(torch.bfloat16)
    check_forward(case, q, k, v)


# Causal grids whose tiles see very different numbers of keys launch in
# chunks of (sequence, query head) units, longest tiles first; these shapes
# leave a short last chunk (32 MiB of K and V per chunk), whose heads are
# among the checked ones.
CHUNKED = [
    (si.fixed("fwd_chunk_d128_b1_h20_s8192_causal", 1, 20, 128, 8192, 8192, True, 211), [(0, 0), (0, 19)]),
    (si.fixed("fwd_chunk_d64_b1_h20_s16384_causal", 1, 20, 64, 16384, 16384, True, 212), [(0, 17)]),
    (si.fixed("fwd_chunk_d256_b1_h6_s8192_causal", 1, 6, 256, 8192, 8192, True, 213), [(0, 1), (0, 5)]),
    (si.fixed("fwd_chunk_gqa_b2_h12_hkv3_s4096_causal", 2, 12, 128, 4096, 4096, True, 214, heads_kv=3),
     [(0, 11), (1, 4)]),
]


@pytest.mark.parametrize("case,subset", CHUNKED, ids=lambda x: getattr(x, "name", "heads"))
def test_forward_chunked_launch_order_sampled(case, subset):
    q, k, v, _ = case.tensors()
    o, m, l = (to_np(t) for t in run_forward(case, q, k, v))
    o64, m64, l64 = oracle.forward_packed(q, k, v, case.cu_q, case.cu_kv, case.softmax_scale, case.causal,
                                          heads_subset=subset)
    for b, h in subset:
        rows = slice(int(case.cu_q[b]), int(case.cu_q[b + 1]))
        compare("O", o[rows, h], o64[rows, h])
        np.testing.assert_allclose(m[rows, h], m64[rows, h], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(l[rows, h], l64[rows, h], rtol=1e-4)
