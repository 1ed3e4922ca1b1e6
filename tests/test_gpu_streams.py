"""The deterministic mode and CUDA streams.  Its two kernels (dK / dV and
dQ) are independent, so the library runs the dQ kernel on a second stream
of the device, forked from and joined back into the caller's stream by
events; under stream capture both run in order on the caller's stream.
Whichever path runs, and whatever else is in flight, the gradients must be
the same bits and the caller's stream must be ordered after both kernels."""
import threading

import pytest
import torch

import seeded_inputs as si
from parity import Prepared, check_case

pytestmark = pytest.mark.gpu

CASES = [
    si.fixed("streams_d128", 2, 4, 128, 1024, 1024, False, 91),
    si.Case("streams_d64_varlen_causal", 4, 64, [300, 1000, 513], [700, 1000, 900], True, 92),
]


def _run(prep, dq_mode, out, work, stream=None, check=True):
    import attention_backward_sm_gb300 as fab
    return fab.backward(prep.q, prep.k, prep.v, prep.o, prep.do, prep.m, prep.l, prep.cu_q, prep.cu_kv,
                        prep.case.cu_q, prep.case.cu_kv, prep.case.causal, prep.scale, dq_mode, out=out,
                        work=work, stream=stream, check=check, **prep.mask_kw)


def _buffers(prep, dq_mode):
    import attention_backward_sm_gb300 as fab
    work = fab.Workspace(prep.q, prep.case.cu_q, prep.case.cu_kv, prep.case.causal, dq_mode)
    out = (torch.empty_like(prep.q), torch.empty_like(prep.k), torch.empty_like(prep.v))
    return out, work


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_deterministic_under_graph_capture(case):
    """A CUDA graph of preprocess -> fa_bwd -> finalize in deterministic
    mode (both kernels on the captured stream) gives the bits of a plain
    call (the dQ kernel on the second stream), replay after replay."""
    import attention_backward_sm_gb300 as fab
    mode = fab.FA_DQ_DETERMINISTIC
    prep = Prepared(case)
    plain = prep.run(dq_mode=mode)
    check_case(prep, out=plain)
    out, work = _buffers(prep, mode)
    _run(prep, mode, out, work)            # warm-up outside the capture
    torch.cuda.synchronize()
    for t in out:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run(prep, mode, out, work, check=False)
    for _ in range(3):
        for t in out:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        fab.fa_check_device_status()
        for a, b in zip(plain, out):
            assert torch.equal(a, b)


def test_deterministic_calls_in_flight_on_two_streams_from_two_threads():
    """Two host threads, each with its own stream and buffers, issue
    deterministic backward calls at the same time (both use the library's
    second stream); every result equals a plain call's bits, and each
    caller's stream is ordered after both of its kernels (the outputs are
    read on that stream right after the call)."""
    import attention_backward_sm_gb300 as fab
    mode = fab.FA_DQ_DETERMINISTIC
    prep = Prepared(CASES[0])
    plain = prep.run(dq_mode=mode)
    n_calls = 20
    sums = {}
    errors = []

    def worker(tid):
        try:
            stream = torch.cuda.Stream()
            out, work = _buffers(prep, mode)
            got = []
            with torch.cuda.stream(stream):
                for _ in range(n_calls):
                    for t in out:
                        t.zero_()
                    _run(prep, mode, out, work, stream=stream, check=False)
                    got.append(tuple(t.clone() for t in out))
            stream.synchronize()
            sums[tid] = got
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    fab.fa_check_device_status()
    for tid, got in sums.items():
        assert len(got) == n_calls
        for res in got:
            for a, b in zip(plain, res):
                assert torch.equal(a, b)


@pytest.mark.parametrize("head_dim", [64, 256])
def test_forward_calls_in_flight_on_two_streams_from_two_threads(head_dim):
    """The one-tile forward (head_dim 64 / 256) from two threads on two
    streams at once: every (O, m, l) equals a plain call's bits."""
    import attention_backward_sm_gb300 as fab
    case = si.fixed(f"streams_fwd_d{head_dim}", 2, 4, head_dim, 1024, 1024, True, 93)
    dev = torch.device("cuda")
    q, k, v, _ = (t.to(dev) for t in case.tensors())
    cu_q = torch.from_numpy(case.cu_q).to(dev)
    cu_kv = torch.from_numpy(case.cu_kv).to(dev)
    plain = fab.forward_stats(q, k, v, cu_q, cu_kv, case.cu_q, case.cu_kv, case.causal, case.softmax_scale)
    results = {}
    errors = []

    def worker(tid):
        try:
            stream = torch.cuda.Stream()
            got = []
            with torch.cuda.stream(stream):
                for _ in range(20):
                    got.append(fab.forward_stats(q, k, v, cu_q, cu_kv, case.cu_q, case.cu_kv, case.causal,
                                                 case.softmax_scale, stream=stream, check=False))
            stream.synchronize()
            results[tid] = got
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    fab.fa_check_device_status()
    for got in results.values():
        for res in got:
            for a, b in zip(plain, res):
                assert torch.equal(a, b)
