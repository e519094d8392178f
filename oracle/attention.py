"""Plain FP64 causal grouped-query attention, forward and backward.

Test infrastructure only (see the package docstring).  Shares nothing with
the CUDA path.

What is computed (TransformerEngine PR "Optimize context parallel attention
layouts and gradient accumulation", Description and Independent-node
complete-CP evidence: "BF16 causal uniform THD", "Hq32/Hkv8", D128/D256).
The pages name the operation without writing it out; the plain textbook
definition is used:

    s_ij  = scale * <q_i, k_j>            for visible keys j (causal: j <= i)
    m_i   = max_j s_ij,   l_i = sum_j exp(s_ij - m_i)
    P_ij  = exp(s_ij - m_i) / l_i
    O_i   = sum_j P_ij v_j,   LSE_i = m_i + ln l_i        (natural log)

    Delta_i = <dO_i, O_i>,   dP_ij = <dO_i, v_j>,   dS_ij = P_ij (dP_ij - Delta_i)
    dQ_i = scale * sum_j dS_ij k_j
    dK_j = scale * sum_i dS_ij q_i,   dV_j = sum_i P_ij dO_i

Readings where the pages are silent:
  * scale = 1/sqrt(D) unless given;
  * GQA: q head h uses kv head floor(h / (Hq/Hkv)) (contiguous groups), and a
    kv head's dK/dV is the sum over the q heads of its group;
  * causal alignment is top-left inside each sequence (query and key lengths
    are equal, so there is no other choice);
  * packed THD with padding: sequence b occupies physical rows
    [cu_seqlens_padded[b], cu_seqlens_padded[b+1]); its first
    S_b = cu_seqlens[b+1]-cu_seqlens[b] rows are real tokens and the rest are
    padding.  Padding rows neither attend nor are attended: their O, dQ, dK,
    dV are 0 and their LSE is -inf.
"""

import numpy as np


def kv_head_of(h, hq, hkv):
    """kv head serving q head ``h`` under contiguous GQA grouping."""
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (hq // hkv)


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def masked_attention(Q, K, V, qpos, kpos, scale):
    """Attention of queries at positions ``qpos`` over keys at ``kpos``.

    A key is visible to a query iff kpos <= qpos (causal by position inside
    one sequence).  Rows that see no key get O = 0 and LSE = -inf.
    Returns (O [nq, D], LSE [nq]) in FP64.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    qpos = np.asarray(qpos)[:, None]
    kpos = np.asarray(kpos)[None, :]
    visible = kpos <= qpos
    S = scale * (Q @ K.T)
    S = np.where(visible, S, -np.inf)
    m = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])          # exp(-inf) = 0 on hidden keys
    l = E.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    P = E / l_safe[:, None]
    O = P @ V
    lse = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    return O, lse


def masked_attention_backward(Q, K, V, dO, qpos, kpos, lse, delta, scale):
    """Gradient contributions of one (query set, key set) block.

    P is rebuilt from the given row LSE (the final, merged one), and
    Delta is the given row dot <dO_i, O_i>.  Returns (dQ [nq,D], dK [nk,D],
    dV [nk,D]) contributions of this block alone.
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    lse = _f64(lse)
    delta = _f64(delta)
    visible = np.asarray(kpos)[None, :] <= np.asarray(qpos)[:, None]
    finite = np.isfinite(lse)
    S = scale * (Q @ K.T)
    P = np.where(visible & finite[:, None],
                 np.exp(S - np.where(finite, lse, 0.0)[:, None]), 0.0)
    dP = dO @ V.T
    dS = P * (dP - delta[:, None])
    dQ = scale * (dS @ K)
    dK = scale * (dS.T @ Q)
    dV = P.T @ dO
    return dQ, dK, dV


def head_forward(Q, K, V, scale=None):
    """Causal attention of one (sequence, q head): O [n,D], LSE [n]."""
    n, D = np.shape(Q)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    pos = np.arange(n)
    return masked_attention(Q, K, V, pos, pos, scale)


def head_backward(Q, K, V, dO, scale=None):
    """Gradients of one (sequence, q head) from its own FP64 forward.

    Returns (dQ, dK, dV, O, LSE); dK and dV are this q head's share of the
    kv head's gradient.
    """
    n, D = np.shape(Q)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O, lse = head_forward(Q, K, V, scale)
    delta = np.sum(_f64(dO) * O, axis=1)
    pos = np.arange(n)
    dQ, dK, dV = masked_attention_backward(Q, K, V, dO, pos, pos, lse, delta, scale)
    return dQ, dK, dV, O, lse


def _sequences(cu_seqlens, cu_seqlens_padded):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cp = np.asarray(cu_seqlens_padded, dtype=np.int64)
    for b in range(len(cu) - 1):
        yield b, int(cp[b]), int(cu[b + 1] - cu[b]), int(cp[b + 1] - cp[b])


def attention_forward(q, k, v, cu_seqlens, cu_seqlens_padded=None, scale=None):
    """Whole packed-THD forward.  q [T,Hq,D], k/v [T,Hkv,D] -> O [T,Hq,D], LSE [T,Hq]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, D = q.shape
    hkv = k.shape[1]
    if cu_seqlens_padded is None:
        cu_seqlens_padded = cu_seqlens
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.zeros((T, hq, D))
    lse = np.full((T, hq), -np.inf)
    for _, start, n, _ in _sequences(cu_seqlens, cu_seqlens_padded):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            o_h, l_h = head_forward(q[start:start + n, h], k[start:start + n, g],
                                    v[start:start + n, g], scale)
            O[start:start + n, h] = o_h
            lse[start:start + n, h] = l_h
    return O, lse


def attention_backward(q, k, v, do, cu_seqlens, cu_seqlens_padded=None, scale=None):
    """Whole packed-THD backward from the oracle's own FP64 forward.

    Returns (dQ [T,Hq,D], dK [T,Hkv,D], dV [T,Hkv,D]); padding rows are 0.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T, hq, D = q.shape
    hkv = k.shape[1]
    if cu_seqlens_padded is None:
        cu_seqlens_padded = cu_seqlens
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for _, start, n, _ in _sequences(cu_seqlens, cu_seqlens_padded):
        sl = slice(start, start + n)
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            dq_h, dk_h, dv_h, _, _ = head_backward(q[sl, h], k[sl, g], v[sl, g],
                                                   do[sl, h], scale)
            dq[sl, h] = dq_h
            dk[sl, g] += dk_h
            dv[sl, g] += dv_h
    return dq, dk, dv
