"""Plain fp64 definition of attention forward statistics and backward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and
by the CPU-baseline leg of ``bench.py``; never by the product path.  It
shares no code with the CUDA library.

Sources (cited by page title and section):
  * "PyPTO-Gym SK-16: single-pass Attention backward (FA Grad)" article
    (czykbl.com news 95943), section 3 (kernel skeleton: C1, V1, C2, V2),
    section 3.1 (the eight per-block steps), section 4.1 (l and m are
    consumed, never recomputed) and section 4.2 (dtype table).
  * JAX ``fused_attention_stablehlo.py``, ``MaskType.CAUSAL`` and the
    backward operand list of ``_dot_product_attention_bwd_cuda_lowering``
    (interface only).
  * PyPTO ``block_attn_res_impl.py`` backward kernel: the softmax-backward
    identity grad_logits = alpha * (grad_alpha - sum(grad_alpha * alpha)).

Every function works on one (sequence, head) with full score matrices in
float64: no tiling, no online softmax, no fused steps.  Inputs are upcast
exactly from their stored types (bf16 / fp32) to float64.

Readings where the pages are silent (each also listed in the design notes):
  * m is the row maximum of the *scaled* scores and l is the plain sum of
    exp(scaled score - m), not a log-sum (section 3.1 step 2 divides by L).
  * scale multiplies the scores before exp and multiplies dQ and dK, not
    dV (section 3, V2: dv is added unscaled, dq and dk are multiplied).
  * D is computed from the O that the backward is given (section 3.1
    step 4, section 4.2 row "D"), not from P @ V.
  * The causal mask is top-left aligned: query i (local index) sees key j
    iff j <= i.  Masked entries have P = 0 exactly.
  * Bottom-right causal (not defined by the pages; the usual alignment of
    the causal diagonal with the last key): query i sees key j iff
    j <= i + (s2 - s1).
  * Sliding window of length W (JAX ``dot_product_attention``,
    ``sliding_window_length``: each token sees the left window
    (pos - W, pos]): query i sees key j iff i + off - W < j <= i + off,
    off = 0 (top-left) or s2 - s1 (bottom-right).  The window carries the
    causal upper bound, so it is only defined together with a causal mask.
  * A row that sees no key (no keys at all, or every key masked) has
    m = -inf, l = 0, O = 0 and dQ = 0.
  * A row with no keys (s2 = 0) has m = -inf, l = 0, O = 0, dQ = 0.
  * No bf16 rounding of P or dS is emulated: the oracle is the exact
    gradient of the stated inputs.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """Exact upcast of a numpy array or a CPU torch tensor to float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: torch is only needed to read torch inputs
        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def visible(s1: int, s2: int, causal: bool, window: int = 0, bottom_right: bool = False) -> np.ndarray:
    """Boolean [s1, s2] matrix: may query i attend to key j.

    Non-causal: every pair.  Causal: j <= i + off, off = 0 for the top-left
    alignment and s2 - s1 for the bottom-right one.  A sliding window of
    length W > 0 (JAX ``dot_product_attention`` ``sliding_window_length``,
    the left window (pos - W, pos]) further requires j > i + off - W."""
    if window < 0:
        raise ValueError("window must be >= 0")
    if (window > 0 or bottom_right) and not causal:
        raise ValueError("a sliding window or the bottom-right alignment needs a causal mask")
    i = np.arange(s1)[:, None]
    j = np.arange(s2)[None, :]
    if not causal:
        return np.ones((s1, s2), dtype=bool)
    off = s2 - s1 if bottom_right else 0
    vis = j <= i + off
    if window > 0:
        vis &= j > i + off - window
    return vis


def masked_scores(q, k, scale: float, causal: bool, window: int = 0, bottom_right: bool = False) -> np.ndarray:
    """X = scale * Q K^T with masked entries set to -inf.

    Section 3.1 steps 1-2 (S = Q K^T, then S * scale); the mask is
    ``visible`` (top-left causal unless told otherwise)."""
    q = _f64(q)
    k = _f64(k)
    x = scale * (q @ k.T)
    return np.where(visible(x.shape[0], x.shape[1], causal, window, bottom_right), x, -np.inf)


def forward_head(q, k, v, scale: float, causal: bool, window: int = 0, bottom_right: bool = False):
    """Forward statistics of one head: (O, m, l), all float64.

    m_i = max_j X_ij, l_i = sum_j exp(X_ij - m_i), P = exp(X - m) / l,
    O = P V.  These are the statistics the SK-16 backward consumes
    (section 3.1 step 2; section 5 says the forward skeleton supplies them).
    Rows that see no key keep m = -inf, l = 0, O = 0.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    s1, d = q.shape
    s2 = k.shape[0]
    o = np.zeros((s1, v.shape[1]))
    m = np.full(s1, -np.inf)
    l = np.zeros(s1)
    if s2 == 0:
        return o, m, l
    x = masked_scores(q, k, scale, causal, window, bottom_right)
    rows = np.isfinite(x).any(axis=1)
    x = x[rows]
    m[rows] = x.max(axis=1)
    e = np.exp(x - m[rows][:, None])
    l[rows] = e.sum(axis=1)
    o[rows] = (e / l[rows][:, None]) @ v
    return o, m, l


def rowsum_o_do(o, do) -> np.ndarray:
    """D_i = sum_k O_ik * dO_ik (section 3.1 step 4)."""
    return (_f64(o) * _f64(do)).sum(axis=1)


def backward_head(q, k, v, o, do, m, l, scale: float, causal: bool, window: int = 0, bottom_right: bool = False):
    """Gradients of one head from the given forward statistics.

    Follows section 3.1 in its order:
      1. S = Q K^T               (with step 2's scale and the mask)
      2. P = exp(S*scale - m) / l   (m, l are inputs, section 4.1)
      3. dP = dO V^T
      4. D = rowsum(O * dO)
      5. dS = P * (dP - D)
      6. dK = scale * dS^T Q
      7. dV = P^T dO
      8. dQ = scale * dS K
    Returns (dQ, dK, dV, D) in float64.
    """
    q, k, v, o, do = (_f64(t) for t in (q, k, v, o, do))
    m, l = _f64(m), _f64(l)
    s1, s2 = q.shape[0], k.shape[0]
    D = rowsum_o_do(o, do)
    if s1 == 0 or s2 == 0:
        return (np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), D)
    x = masked_scores(q, k, scale, causal, window, bottom_right)
    # P is 0 at masked entries; rows that see no key (l = 0) are all 0
    rows = l > 0
    p = np.zeros_like(x)
    p[rows] = np.exp(x[rows] - m[rows][:, None]) / l[rows][:, None]
    dp = do @ v.T
    ds = p * (dp - D[:, None])
    dk = scale * (ds.T @ q)
    dv = p.T @ do
    dq = scale * (ds @ k)
    return dq, dk, dv, D


def _kv_head(h: int, hq: int, hkv: int) -> int:
    """Key/value head used by query head h when hq query heads share hkv
    key/value heads in equal consecutive groups (grouped-query attention,
    the JAX cuDNN wrapper's q_N != kv_N case; hkv = hq is plain multi-head,
    hkv = 1 is multi-query)."""
    if hq % hkv != 0:
        raise ValueError(f"query heads ({hq}) must be a multiple of key/value heads ({hkv})")
    return h // (hq // hkv)


def forward_packed(q, k, v, cu_q, cu_kv, scale: float, causal: bool,
                   heads_subset=None, window: int = 0, bottom_right: bool = False):
    """Forward statistics over a packed batch ``[total, H, d]``.

    cu_q / cu_kv are the cumulative offsets (``actual_q`` / ``actual_kv``,
    section 3).  Rows outside every sequence are left at O = 0, m = -inf,
    l = 0.  ``heads_subset`` restricts the work to a list of (b, h) pairs.
    K and V may have fewer heads than Q (grouped-query attention).
    Returns float64 arrays O [total_q, H, d], m and l [total_q, H].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_kv = np.asarray(cu_kv, dtype=np.int64)
    total_q, H, d = q.shape
    Hkv = k.shape[1]
    o = np.zeros((total_q, H, v.shape[2]))
    m = np.full((total_q, H), -np.inf)
    l = np.zeros((total_q, H))
    units = heads_subset if heads_subset is not None else [
        (b, h) for b in range(len(cu_q) - 1) for h in range(H)]
    for b, h in units:
        qs, qe = cu_q[b], cu_q[b + 1]
        ks, ke = cu_kv[b], cu_kv[b + 1]
        hk = _kv_head(h, H, Hkv)
        ob, mb, lb = forward_head(q[qs:qe, h], k[ks:ke, hk], v[ks:ke, hk], scale, causal, window, bottom_right)
        o[qs:qe, h], m[qs:qe, h], l[qs:qe, h] = ob, mb, lb
    return o, m, l


def lse_from_stats(m, l) -> np.ndarray:
    """The single softmax statistic lse_i = log(sum_j exp(X_ij)) = m_i + log(l_i)
    (natural log; -inf for rows that see no key).  JAX's cuDNN wrapper keeps
    one float32 ``softmax_stat`` per query row between forward and backward;
    this is the reading of what it holds."""
    m, l = _f64(m), _f64(l)
    out = np.full(m.shape, -np.inf)
    rows = l > 0
    out[rows] = m[rows] + np.log(l[rows])
    return out


def backward_head_lse(q, k, v, o, do, lse, scale: float, causal: bool, window: int = 0,
                      bottom_right: bool = False):
    """backward_head with P = exp(X - lse) from the single statistic lse
    instead of exp(X - m) / l; the other steps are the same."""
    q, k, v, o, do = (_f64(t) for t in (q, k, v, o, do))
    lse = _f64(lse)
    s1, s2 = q.shape[0], k.shape[0]
    D = rowsum_o_do(o, do)
    if s1 == 0 or s2 == 0:
        return (np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), D)
    x = masked_scores(q, k, scale, causal, window, bottom_right)
    rows = np.isfinite(lse)
    p = np.zeros_like(x)
    p[rows] = np.exp(x[rows] - lse[rows][:, None])
    dp = do @ v.T
    ds = p * (dp - D[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), p.T @ do, D


def backward_packed_lse(q, k, v, o, do, lse, cu_q, cu_kv, scale: float, causal: bool, heads_subset=None,
                        window: int = 0, bottom_right: bool = False):
    """backward_packed from lse [total_q, H] instead of (m, l)."""
    q, k, v, o, do = (_f64(t) for t in (q, k, v, o, do))
    lse = _f64(lse)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_kv = np.asarray(cu_kv, dtype=np.int64)
    H, Hkv = q.shape[1], k.shape[1]
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    D = np.zeros(q.shape[:2])
    units = heads_subset if heads_subset is not None else [
        (b, h) for b in range(len(cu_q) - 1) for h in range(H)]
    for b, h in units:
        qs, qe = cu_q[b], cu_q[b + 1]
        ks, ke = cu_kv[b], cu_kv[b + 1]
        hk = _kv_head(h, H, Hkv)
        r = backward_head_lse(q[qs:qe, h], k[ks:ke, hk], v[ks:ke, hk], o[qs:qe, h], do[qs:qe, h],
                              lse[qs:qe, h], scale, causal, window, bottom_right)
        dq[qs:qe, h], D[qs:qe, h] = r[0], r[3]
        dk[ks:ke, hk] += r[1]
        dv[ks:ke, hk] += r[2]
    return dq, dk, dv, D


def backward_packed(q, k, v, o, do, m, l, cu_q, cu_kv, scale: float,
                    causal: bool, heads_subset=None, window: int = 0, bottom_right: bool = False):
    """Backward over a packed batch from the given (O, m, l).

    Returns float64 dQ [total_q,H,d], dK and dV [total_kv,Hkv,d] and
    D [total_q,H].  Rows outside every sequence (padding) are exactly 0.
    With grouped-query attention (K, V with Hkv < H heads) the gradient of a
    shared key/value head is the sum over the query heads of its group.
    """
    q, k, v, o, do = (_f64(t) for t in (q, k, v, o, do))
    m, l = _f64(m), _f64(l)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_kv = np.asarray(cu_kv, dtype=np.int64)
    H = q.shape[1]
    Hkv = k.shape[1]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    D = np.zeros(q.shape[:2])
    units = heads_subset if heads_subset is not None else [
        (b, h) for b in range(len(cu_q) - 1) for h in range(H)]
    for b, h in units:
        qs, qe = cu_q[b], cu_q[b + 1]
        ks, ke = cu_kv[b], cu_kv[b + 1]
        hk = _kv_head(h, H, Hkv)
        r = backward_head(q[qs:qe, h], k[ks:ke, hk], v[ks:ke, hk], o[qs:qe, h],
                          do[qs:qe, h], m[qs:qe, h], l[qs:qe, h], scale, causal, window, bottom_right)
        dq[qs:qe, h], D[qs:qe, h] = r[0], r[3]
        dk[ks:ke, hk] += r[1]
        dv[ks:ke, hk] += r[2]
    return dq, dk, dv, D
