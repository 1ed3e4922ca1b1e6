"""GPU parity on problems whose packed tensors hold more than 2^31 elements
(every element offset past that point must be computed in 64 bits): the GPU
runs the whole problem, the fp64 oracle checks the last (sequence, head)
unit, which lies beyond the 2^31-th element of every [rows, heads, d]
tensor.  Inputs are drawn on the device by a seeded generator; the checked
unit's slices are copied to the host for the oracle."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity import compare, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # 260 x 4096 rows, 16 heads, d = 128: 2.18e9 elements per tensor
    (260, 4096, 16, 128, True, 1201),
    # the head_dim 256 kernel: 260 x 4096 rows, 8 heads
    (260, 4096, 8, 256, False, 1202),
]


@pytest.mark.parametrize("batch,s,heads,d,causal,seed", CASES, ids=["d128_causal", "d256_noncausal"])
def test_beyond_2e31_elements(batch, s, heads, d, causal, seed):
    import attention_backward_sm_gb300 as fab
    need = 11 * batch * s * heads * d * 2   # 8 bf16 tensors, the fp32 dQ accumulator, statistics
    if torch.cuda.get_device_properties(0).total_memory < 1.5 * need:
        pytest.skip("device memory too small for this size")
    total = batch * s
    assert total * heads * d > 2**31
    cu = si.cumulative([s] * batch)
    cu_dev = torch.from_numpy(cu).cuda()
    shape = (total, heads, d)
    q, k, v, do = (si.bf16_normal_device(shape, seed, sub) for sub in range(4))
    scale = d ** -0.5
    b, h = batch - 1, heads - 1                  # the checked unit: last sequence, last head
    rows = slice(int(cu[b]), int(cu[b + 1]))
    assert int(cu[b]) * heads * d + h * d > 2**31
    # forward statistics: the library's for every unit, the oracle's for the checked one
    o, m, l = fab.forward_stats(q, k, v, cu_dev, cu_dev, cu, cu, causal, scale)
    one = np.array([0, s], dtype=np.int32)
    qs, ks, vs, dos = (t[rows].cpu() for t in (q, k, v, do))
    o64, m64, l64 = oracle.forward_packed(qs, ks, vs, one, one, scale, causal, heads_subset=[(0, h)])
    o_u = torch.from_numpy(o64).to(torch.bfloat16)
    m_u = torch.from_numpy(m64).to(torch.float32)
    l_u = torch.from_numpy(l64).to(torch.float32)
    o[rows, h] = o_u[:, h].cuda()
    m[rows, h] = m_u[:, h].cuda()
    l[rows, h] = l_u[:, h].cuda()
    dq, dk, dv = fab.backward(q, k, v, o, do, m, l, cu_dev, cu_dev, cu, cu, causal, scale)
    torch.cuda.synchronize()
    fab.fa_check_device_status()
    ref = oracle.backward_packed(qs, ks, vs, o_u, dos, m_u, l_u, one, one, scale, causal, heads_subset=[(0, h)])
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref[:3]):
        compare(name, to_np(g[rows, h]), r[:, h])
    # the last rows of every output were written (finite, not all zero)
    for t in (dq, dk, dv):
        tail = t[-8:].float()
        assert torch.isfinite(tail).all() and tail.abs().sum() > 0
    del q, k, v, do, o, m, l, dq, dk, dv
    torch.cuda.empty_cache()
