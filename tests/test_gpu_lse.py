"""GPU parity of the single-statistic path (fa_fwd_lse, fa_bwd_lse:
lse = m + ln l, the reading of JAX's float32 softmax_stat) against the fp64
oracle's lse backward."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity import Prepared, check_case, to_np

pytestmark = pytest.mark.gpu


CASES = [
    si.fixed("lse_d128_noncausal", 2, 3, 128, 300, 333, False, 101),
    si.fixed("lse_d64_causal", 1, 4, 64, 517, 517, True, 102),
    si.Case("lse_varlen_gqa_br_window_d128", 4, 128, [100, 0, 700, 5], [250, 9, 300, 5], True, 103, pad_q=3,
            pad_kv=4, heads_kv=2, bottom_right=True, window=190),
]


class LsePrepared(Prepared):
    """Prepared with lse = m + ln l (fp64 from the oracle statistics, then
    fp32) fed to fa_bwd_lse and to the oracle's lse backward."""

    def __init__(self, case, **kw):
        super().__init__(case, **kw)
        self.lse_cpu = torch.from_numpy(oracle.lse_from_stats(self.m_cpu, self.l_cpu)).to(torch.float32)
        self.lse = self.lse_cpu.to(self.q.device)

    def reference(self):
        q, k, v, do = self.cpu
        return oracle.backward_packed_lse(q, k, v, self.o_cpu, do, self.lse_cpu, self.case.cu_q, self.case.cu_kv,
                                          self.scale, self.case.causal, heads_subset=self.heads_subset,
                                          **self.mask_kw)

    def run(self, dq_mode=0):
        import attention_backward_sm_gb300 as fab
        out = fab.backward_lse(self.q, self.k, self.v, self.o, self.do, self.lse, self.cu_q, self.cu_kv,
                               self.case.cu_q, self.case.cu_kv, self.case.causal, self.scale, dq_mode,
                               **self.mask_kw)
        torch.cuda.synchronize()
        fab.fa_check_device_status()
        return out


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_lse_backward_parity(case):
    import attention_backward_sm_gb300 as fab
    prep = LsePrepared(case)
    check_case(prep)
    check_case(prep, out=prep.run(fab.FA_DQ_DETERMINISTIC))


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_lse_forward(case):
    """fa_fwd_lse: O as the oracle forward, lse = m + ln l of the oracle
    statistics (-inf exactly for rows that see no key)."""
    import attention_backward_sm_gb300 as fab
    prep = LsePrepared(case)
    o, lse = fab.forward_lse(prep.q, prep.k, prep.v, prep.cu_q, prep.cu_kv, case.cu_q, case.cu_kv, case.causal,
                             prep.scale, window=case.window, bottom_right=case.bottom_right)
    torch.cuda.synchronize()
    n = int(case.cu_q[-1])
    ref_o = prep.o_cpu.double().numpy()[:n]
    ref = oracle.lse_from_stats(prep.m_cpu, prep.l_cpu)[:n]
    got = to_np(lse)[:n]
    assert np.abs(to_np(o)[:n] - ref_o).max() <= 2e-2 * np.abs(ref_o).max()
    empty = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), empty)
    assert np.allclose(got[~empty], ref[~empty], rtol=1e-5, atol=1e-5)
