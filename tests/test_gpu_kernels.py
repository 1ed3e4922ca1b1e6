"""GPU parity of the support and bandwidth-bound steps against the oracle:
fa_fwd_stats (O, m, l), fa_bwd_preprocess (D and the zeroed accumulator),
fa_bwd_dq_finalize, and the status / error paths through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity import compare, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    si.cfg1(),
    si.fixed("fwd_d128_causal_tail", 2, 3, 128, 300, 300, True, 31),
    si.Case("fwd_varlen_cross_d64", 2, 64, [70, 0, 129], [200, 9, 0], False, 32, pad_q=3, pad_kv=2),
    si.Case("fwd_varlen_causal_d128", 2, 128, [190, 64], [150, 64], True, 33),
], ids=lambda c: c.name)
def test_fwd_stats(case):
    import attention_backward_sm_gb300 as fab
    q, k, v, _ = case.tensors()
    o64, m64, l64 = oracle.forward_packed(q, k, v, case.cu_q, case.cu_kv, case.softmax_scale, case.causal)
    dev = torch.device("cuda")
    cu_q, cu_kv = torch.from_numpy(case.cu_q).to(dev), torch.from_numpy(case.cu_kv).to(dev)
    o, m, l = fab.forward_stats(q.to(dev), k.to(dev), v.to(dev), cu_q, cu_kv, case.cu_q, case.cu_kv, case.causal,
                                case.softmax_scale)
    torch.cuda.synchronize()
    nq = int(case.cu_q[-1])
    o, m, l = to_np(o)[:nq], to_np(m)[:nq], to_np(l)[:nq]
    compare("O", o, o64[:nq])
    fin = np.isfinite(m64[:nq])
    assert np.array_equal(np.isfinite(m), fin)
    np.testing.assert_allclose(m[fin], m64[:nq][fin], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(l, l64[:nq], rtol=1e-4, atol=0)


@pytest.mark.parametrize("d", [64, 128])
def test_preprocess_and_finalize(d):
    import attention_backward_sm_gb300 as fab
    case = si.fixed("pre", 1, 3, d, 1000, 1000, False, 41)
    q, k, v, do = case.tensors()
    o = si.bf16_normal(q.shape, 42)
    dev = torch.device("cuda")
    D = torch.full((1000, 3), float("nan"), device=dev)
    acc = torch.full((1000, 3, d), float("nan"), device=dev)
    fab.fa_bwd_preprocess(o.to(dev), do.to(dev), D, acc)
    torch.cuda.synchronize()
    assert torch.count_nonzero(acc).item() == 0
    want = np.stack([oracle.rowsum_o_do(o[:, h], do[:, h]) for h in range(o.shape[1])], axis=1)
    np.testing.assert_allclose(to_np(D), want, rtol=1e-5, atol=1e-4)
    x = torch.randn(1000, 3, d, device=dev)
    dq = torch.empty(1000, 3, d, dtype=torch.bfloat16, device=dev)
    fab.fa_bwd_dq_finalize(x, dq, 0.125)
    torch.cuda.synchronize()
    # exact: bf16 round-to-nearest-even of (0.125 * x), a power-of-two scaling
    assert torch.equal(dq.cpu(), (x * 0.125).to(torch.bfloat16).cpu())


def test_unsupported_head_dim_raises():
    import attention_backward_sm_gb300 as fab
    case = si.fixed("bad", 1, 1, 64, 16, 16, False, 1)
    q = torch.zeros(16, 1, 96, dtype=torch.bfloat16, device="cuda")
    cu = torch.from_numpy(case.cu_q).cuda()
    with pytest.raises(fab.FabwdError) as e:
        fab.forward_stats(q, q, q, cu, cu, case.cu_q, case.cu_kv, False, 0.1)
    assert e.value.code == fab.FA_ERR_UNSUPPORTED


def test_device_status_clean_after_runs():
    import attention_backward_sm_gb300 as fab
    fab.fa_check_device_status()


def test_bounded_wait_times_out_into_a_status_code():
    """A wait that nothing satisfies ends after its limit with FA_ERR_TIMEOUT
    in the status word (no trap, no hang), and the context stays usable: a
    backward right after runs and reports a clean status."""
    import attention_backward_sm_gb300 as fab
    fab.fa_check_device_status()
    fab.fa_selftest_wait_timeout()
    with pytest.raises(fab.FabwdError) as e:
        fab.fa_check_device_status()
    assert e.value.code == fab.FA_ERR_TIMEOUT
    fab.fa_check_device_status()                # the word was cleared
    case = si.fixed("after_timeout", 1, 2, 128, 200, 200, True, 43)
    q, k, v, do = (t.cuda() for t in case.tensors())
    cu = torch.from_numpy(case.cu_q).cuda()
    o, m, l = fab.forward_stats(q, k, v, cu, cu, case.cu_q, case.cu_kv, True, case.softmax_scale)
    dq, dk, dv = fab.backward(q, k, v, o, do, m, l, cu, cu, case.cu_q, case.cu_kv, True, case.softmax_scale)
    torch.cuda.synchronize()
    fab.fa_check_device_status()
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dk.float()).all()
