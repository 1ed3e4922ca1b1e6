"""Shared helpers of the GPU parity tests: inputs, oracle references and the
comparison rule.

The rule for every gradient (the target specification): relative L2 error
<= 1e-2 and max |error| <= 3e-2 * max |reference| against the fp64 oracle,
and the GPU value exactly 0 wherever the oracle is exactly 0 (padding rows,
keys no query sees).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

REL_L2 = 1e-2
MAX_ABS = 3e-2


def structural_zero_rows(case: si.Case):
    """Rows whose gradients are exactly zero by construction, independent of
    rounding: padding rows, queries that see no key and keys that no query
    sees (the oracle's visibility rule for the case's mask)."""
    zq = np.zeros(case.total_q, dtype=bool)
    zk = np.zeros(case.total_kv, dtype=bool)
    zq[int(case.cu_q[-1]):] = True
    zk[int(case.cu_kv[-1]):] = True
    for b in range(case.batch):
        q0, q1 = int(case.cu_q[b]), int(case.cu_q[b + 1])
        k0, k1 = int(case.cu_kv[b]), int(case.cu_kv[b + 1])
        vis = oracle.visible(q1 - q0, k1 - k0, case.causal, case.window, case.bottom_right)
        zq[q0:q1] = ~vis.any(axis=1)
        zk[k0:k1] = ~vis.any(axis=0)
    return zq, zk


def compare(name, got, ref, exact_zero_mask=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    nref = np.linalg.norm(ref)
    if nref == 0:
        assert np.all(got == 0), f"{name}: reference is all zero, GPU is not"
        return 0.0
    rel = np.linalg.norm(got - ref) / nref
    mx = np.abs(got - ref).max()
    assert rel <= REL_L2, f"{name}: relative L2 error {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS * np.abs(ref).max(), f"{name}: max abs error {mx:.3e} > {MAX_ABS} * {np.abs(ref).max():.3e}"
    if exact_zero_mask is not None:
        bad = np.count_nonzero(got[exact_zero_mask] != 0)
        assert bad == 0, f"{name}: {bad} non-zero values where the result must be exactly 0"
    return rel


def to_np(t):
    return t.detach().float().cpu().double().numpy()


class Prepared:
    """Device copies of one case's inputs with O, m, l for the checked heads
    taken from the oracle forward (rounded to bf16 / fp32).  Heads that are
    not checked use the library's forward statistics."""

    def __init__(self, case: si.Case, heads_subset=None, device="cuda"):
        import attention_backward_sm_gb300 as fab
        self.case = case
        self.heads_subset = heads_subset
        q, k, v, do = case.tensors()
        self.cpu = (q, k, v, do)
        self.scale = case.softmax_scale
        dev = torch.device(device)
        self.cu_q = torch.from_numpy(case.cu_q).to(dev)
        self.cu_kv = torch.from_numpy(case.cu_kv).to(dev)
        self.q, self.k, self.v, self.do = (t.to(dev) for t in (q, k, v, do))
        self.mask_kw = dict(window=case.window, bottom_right=case.bottom_right)
        o64, m64, l64 = oracle.forward_packed(q, k, v, case.cu_q, case.cu_kv, self.scale, case.causal,
                                              heads_subset=heads_subset, **self.mask_kw)
        o = torch.from_numpy(o64).to(torch.bfloat16)
        m = torch.from_numpy(m64).to(torch.float32)
        l = torch.from_numpy(l64).to(torch.float32)
        if heads_subset is None:
            self.o, self.m, self.l = o.to(dev), m.to(dev), l.to(dev)
        else:
            self.o, self.m, self.l = fab.forward_stats(self.q, self.k, self.v, self.cu_q, self.cu_kv, case.cu_q,
                                                       case.cu_kv, case.causal, self.scale, **self.mask_kw)
            for b, h in heads_subset:
                rows = slice(int(case.cu_q[b]), int(case.cu_q[b + 1]))
                self.o[rows, h] = o[rows, h].to(dev)
                self.m[rows, h] = m[rows, h].to(dev)
                self.l[rows, h] = l[rows, h].to(dev)
        self.o_cpu = o
        self.m_cpu = m
        self.l_cpu = l

    def reference(self):
        q, k, v, do = self.cpu
        return oracle.backward_packed(q, k, v, self.o_cpu, do, self.m_cpu, self.l_cpu, self.case.cu_q,
                                      self.case.cu_kv, self.scale, self.case.causal,
                                      heads_subset=self.heads_subset, **self.mask_kw)

    def run(self, dq_mode=0):
        import attention_backward_sm_gb300 as fab
        out = fab.backward(self.q, self.k, self.v, self.o, self.do, self.m, self.l, self.cu_q, self.cu_kv,
                           self.case.cu_q, self.case.cu_kv, self.case.causal, self.scale, dq_mode, **self.mask_kw)
        torch.cuda.synchronize()
        fab.fa_check_device_status()
        return out


def check_case(prep: Prepared, out=None, dq_mode=0):
    """Compares the GPU gradients with the oracle on the checked heads."""
    dq, dk, dv = out if out is not None else prep.run(dq_mode)
    ref = prep.reference()
    case = prep.case
    units = prep.heads_subset or [(b, h) for b in range(case.batch) for h in range(case.heads)]
    got = (to_np(dq), to_np(dk), to_np(dv))
    errs = {}
    zq, zk = structural_zero_rows(case)
    if prep.heads_subset is None:
        for name, g, r, z in zip(("dq", "dk", "dv"), got, ref[:3], (zq, zk, zk)):
            errs[name] = compare(name, g, r, np.broadcast_to(z[:, None, None], g.shape))
    else:
        # dQ per checked (sequence, query head); dK/dV per (sequence, key/value
        # head) whose whole group of query heads is checked (with grouped-query
        # attention a key/value head's gradient sums over its group).
        G = case.heads // case.kv_heads
        for b, h in units:
            qr = slice(int(case.cu_q[b]), int(case.cu_q[b + 1]))
            gg = got[0][qr, h]
            errs[f"dq[{b},{h}]"] = compare(f"dq[b={b},h={h}]", gg, ref[0][qr, h],
                                           np.broadcast_to(zq[qr][:, None], gg.shape))
        checked = set(units)
        groups = sorted({(b, h // G) for b, h in units
                         if all((b, h // G * G + i) in checked for i in range(G))})
        assert groups, "no complete group of query heads among the checked units"
        for b, hk in groups:
            kr = slice(int(case.cu_kv[b]), int(case.cu_kv[b + 1]))
            for name, g, r in zip(("dk", "dv"), got[1:], ref[1:3]):
                gg = g[kr, hk]
                errs[f"{name}[{b},{hk}]"] = compare(f"{name}[b={b},hkv={hk}]", gg, r[kr, hk],
                                                    np.broadcast_to(zk[kr][:, None], gg.shape))
    # structural zeros hold for every head, checked or not
    for g, z in ((got[0], zq), (got[1], zk), (got[2], zk)):
        assert np.all(g[z] == 0), "non-zero gradient in a padding row or a row no query/key reaches"
    return errs
