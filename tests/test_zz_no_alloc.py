"""fa_bwd_noalloc: the backward for callers that cannot allocate device
memory (a runtime that plans all device memory itself, a serving loop in
which an allocation would stall the device, a fixed memory budget).  It
must give the same gradients as the ordinary entry points, which take
their scratch buffers from the caller, and match the fp64 oracle, on two
calls in a row: the fixed scratch array keeps the previous call's
contents, so the second call checks that everything that must start at
zero is cleared again.

This file is collected last on purpose: a failure here leaves every other
test already run."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity import Prepared, check_case, compare, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    si.fixed("noalloc_d128_causal_tail", 2, 4, 128, 300, 300, True, 71),
    si.Case("noalloc_d64_varlen_cross", 3, 64, [130, 1, 257], [200, 64, 129], False, 72, pad_q=3, pad_kv=5),
    si.fixed("noalloc_d256_causal_tail", 1, 2, 256, 200, 200, True, 74),
], ids=lambda c: c.name)
def test_noalloc_matches_entry_points_and_oracle_twice(case):
    import attention_backward_sm_gb300 as fab
    # O, m, l from the oracle forward, so that both sides see the oracle's inputs
    prep = Prepared(case)
    ref_dq, ref_dk, ref_dv = prep.run()
    for call in range(2):
        dq = torch.full_like(prep.q, float("nan"))
        dk = torch.full_like(prep.k, float("nan"))
        dv = torch.full_like(prep.v, float("nan"))
        fab.fa_bwd_noalloc(prep.q, prep.k, prep.v, prep.o, prep.do, prep.m, prep.l, dq, dk, dv, prep.cu_q,
                           prep.cu_kv, case.cu_q, case.cu_kv, case.causal, prep.scale)
        torch.cuda.synchronize()
        fab.fa_check_device_status()
        # against the ordinary entry points: dK and dV are written once per
        # key block without atomics (identical bits); dQ sums fp32 partials
        # with atomics in any order (the parity tolerance)
        assert torch.equal(dk, ref_dk), f"call {call}: dk differs"
        assert torch.equal(dv, ref_dv), f"call {call}: dv differs"
        compare(f"dq (call {call})", to_np(dq), to_np(ref_dq))
        nq = int(case.cu_q[-1])
        assert torch.count_nonzero(dq[nq:]).item() == 0
        # against the fp64 oracle, element by element
        check_case(prep, out=(dq, dk, dv))


def test_noalloc_rejects_problems_beyond_the_fixed_scratch():
    import attention_backward_sm_gb300 as fab
    heads, d = 16, 128
    total = (16 * 1024 * 1024) // (heads * (d + 1) * 4) + 1
    case = si.fixed("noalloc_too_big", 1, heads, d, total, 8, False, 73)
    dev = torch.device("cuda")
    q = torch.zeros(total, heads, d, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(8, heads, d, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(total, heads, dtype=torch.float32, device=dev)
    cu_q, cu_kv = torch.from_numpy(case.cu_q).to(dev), torch.from_numpy(case.cu_kv).to(dev)
    with pytest.raises(fab.FabwdError) as e:
        fab.fa_bwd_noalloc(q, kv, kv, q, q, st, st, q, kv, kv, cu_q, cu_kv, case.cu_q, case.cu_kv, False, 0.1)
    assert e.value.code == fab.FA_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
