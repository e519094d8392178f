"""Context-parallel decomposition of causal attention, FP64 CPU.

Test infrastructure only (see the package docstring).  Shares nothing with
the CUDA path.

Sources (TransformerEngine PR "Optimize context parallel attention layouts
and gradient accumulation"):
  * Changes / CP8 first-gradient accumulator reuse: the first dK/dV
    contribution already holds the accumulator's initial value and is used
    as the accumulator; later additions, their order and the reorder are
    unchanged.
  * Description: per-rank partial outputs carry LSE ("Stats") and are
    combined by the CP algorithm (LSE correction).
  * Independent-node complete-CP evidence: CP8 over B64/S8192 packed THD,
    i.e. each sequence is cut into 2*CP chunks with rank r holding chunks
    r and 2CP-1-r (the load-balanced causal split that the page's "reorder"
    refers to).

Readings where the pages are silent (the same readings as the CUDA path):
  * chunks are cut on the PADDED length P_b (P_b % 2CP must be 0); chunk c
    of sequence b covers physical rows [start_b + c*L_b, start_b+(c+1)*L_b),
    L_b = P_b / (2CP);
  * ring (P2P) exchange: at step s rank r attends with the KV of rank
    src = (r - s) mod CP; the step's partial is attention of r's query
    chunks over src's two KV chunks under the global causal mask;
  * partials merge in ascending step order s = 0..CP-1;
  * backward P uses the final merged LSE and Delta uses the merged O;
  * dQ of a query chunk accumulates over steps s ascending, KV chunk
    ascending inside a step;
  * dK/dV of a KV chunk j (owned by rank src) accumulate contributions from
    ranks src, src+1, ... (mod CP), i.e. ring steps s = 0..CP-1; inside one
    contribution the query chunk r comes before 2CP-1-r, then q heads of the
    GQA group ascending.  The first contribution (step 0, the diagonal one)
    becomes the accumulator: acc = c_0; acc = acc + c_1; ...
"""

import numpy as np

from .attention import masked_attention, masked_attention_backward, kv_head_of


def chunk_owner(c, cp):
    """Rank holding chunk ``c`` of a sequence cut into 2*cp chunks."""
    return c if c < cp else 2 * cp - 1 - c


def rank_chunks(r, cp):
    """The two chunks rank ``r`` holds: the early one r and the late one 2cp-1-r."""
    return (r, 2 * cp - 1 - r)


def ring_source(r, s, cp):
    """Rank whose KV rank ``r`` attends with at ring step ``s``."""
    return (r - s) % cp


def visible_kv_chunks(cq, src, cp):
    """KV chunks of rank ``src`` that query chunk ``cq`` sees (causal: j <= cq)."""
    return [j for j in rank_chunks(src, cp) if j <= cq]


def partial_steps_for_chunk(c, cp):
    """Ring steps at which query chunk ``c`` produces a partial output."""
    r = chunk_owner(c, cp)
    return [s for s in range(cp) if visible_kv_chunks(c, ring_source(r, s, cp), cp)]


def chunk_table(cu_seqlens_padded, cp):
    """[B, 2cp, 2] int64 table of (first physical row, length) per chunk."""
    cpad = np.asarray(cu_seqlens_padded, dtype=np.int64)
    C = 2 * cp
    B = len(cpad) - 1
    tab = np.zeros((B, C, 2), dtype=np.int64)
    for b in range(B):
        P = int(cpad[b + 1] - cpad[b])
        if P % C:
            raise ValueError(f"padded length {P} of sequence {b} is not a multiple of 2*CP={C}")
        L = P // C
        for c in range(C):
            tab[b, c] = (cpad[b] + c * L, L)
    return tab


def _chunk_rows(tab, b, c, seqlen, start):
    """Physical rows and in-sequence positions of the REAL tokens of chunk c."""
    c0, L = int(tab[b, c, 0]), int(tab[b, c, 1])
    pos = np.arange(c0 - start, c0 - start + L)
    pos = pos[pos < seqlen]
    return start + pos, pos


def _seq_info(cu_seqlens, cu_seqlens_padded):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cpad = np.asarray(cu_seqlens_padded, dtype=np.int64)
    return [(int(cpad[b]), int(cu[b + 1] - cu[b])) for b in range(len(cu) - 1)]


def cp_forward_partials(q, k, v, cu_seqlens, cu_seqlens_padded, cp, scale=None):
    """Per-step partials of the ring schedule.

    Returns a list over steps s of (O_s [T,Hq,D], LSE_s [T,Hq]).  A row with no
    partial at step s (an early chunk whose source rank holds only later KV,
    or a padding row) has O_s = 0 and LSE_s = -inf.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T, hq, D = q.shape
    hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    tab = chunk_table(cu_seqlens_padded, cp)
    seqs = _seq_info(cu_seqlens, cu_seqlens_padded)
    parts = []
    for s in range(cp):
        O = np.zeros((T, hq, D))
        lse = np.full((T, hq), -np.inf)
        for b, (start, n) in enumerate(seqs):
            for r in range(cp):
                src = ring_source(r, s, cp)
                for cq in rank_chunks(r, cp):
                    vis = visible_kv_chunks(cq, src, cp)
                    if not vis:
                        continue
                    qrows, qpos = _chunk_rows(tab, b, cq, n, start)
                    kr = [_chunk_rows(tab, b, j, n, start) for j in vis]
                    krows = np.concatenate([x[0] for x in kr])
                    kpos = np.concatenate([x[1] for x in kr])
                    if len(qrows) == 0:
                        continue
                    for h in range(hq):
                        g = kv_head_of(h, hq, hkv)
                        o_h, l_h = masked_attention(q[qrows, h], k[krows, g], v[krows, g],
                                                    qpos, kpos, scale)
                        O[qrows, h] = o_h
                        lse[qrows, h] = l_h
        parts.append((O, lse))
    return parts


def lse_merge(parts):
    """K-way merge of partial (O_s, LSE_s) in the given (step) order.

    M = max_s LSE_s;  sigma = sum_s exp(LSE_s - M);  LSE = M + ln sigma;
    O = sum_s exp(LSE_s - LSE) * O_s.  Rows whose partials are all -inf get
    O = 0 and LSE = -inf.
    """
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])
    M = lses.max(axis=0)
    empty = ~np.isfinite(M)
    M_safe = np.where(empty, 0.0, M)
    sigma = np.exp(lses - M_safe[None]).sum(axis=0)
    lse = np.where(empty, -np.inf, M_safe + np.log(np.where(empty, 1.0, sigma)))
    lse_safe = np.where(empty, 0.0, lse)
    O = np.zeros_like(np.asarray(parts[0][0], dtype=np.float64))
    for O_s, l_s in parts:
        w = np.where(empty, 0.0, np.exp(np.asarray(l_s, dtype=np.float64) - lse_safe))
        O = O + w[..., None] * np.asarray(O_s, dtype=np.float64)
    return O, lse


def cp_attention_forward(q, k, v, cu_seqlens, cu_seqlens_padded, cp, scale=None):
    """CP-emulated forward: ring partials, then the K-way LSE merge."""
    return lse_merge(cp_forward_partials(q, k, v, cu_seqlens, cu_seqlens_padded, cp, scale))


def dq_contribution_order(cq, cp):
    """(step, kv chunk) pairs feeding query chunk ``cq``'s dQ, in order."""
    r = chunk_owner(cq, cp)
    out = []
    for s in range(cp):
        for j in visible_kv_chunks(cq, ring_source(r, s, cp), cp):
            out.append((s, j))
    return out


def dkdv_contribution_order(j, cp):
    """(step, rank, query chunk) triples feeding KV chunk ``j``'s dK/dV, in order.

    The first triple is the step-0 diagonal contribution, which becomes the
    accumulator.
    """
    src = chunk_owner(j, cp)
    out = []
    for s in range(cp):
        r = (src + s) % cp
        for cq in rank_chunks(r, cp):
            if j <= cq:
                out.append((s, r, cq))
    return out


def cp_attention_backward(q, k, v, do, cu_seqlens, cu_seqlens_padded, cp, scale=None):
    """CP-emulated backward in the canonical fixed order.

    Uses the oracle's own CP forward (merged O and LSE), Delta = <dO, O>.
    Returns (dQ, dK, dV) in FP64.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    T, hq, D = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O, lse = cp_attention_forward(q, k, v, cu_seqlens, cu_seqlens_padded, cp, scale)
    delta = np.sum(do * O, axis=2)
    tab = chunk_table(cu_seqlens_padded, cp)
    seqs = _seq_info(cu_seqlens, cu_seqlens_padded)
    C = 2 * cp
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, (start, n) in enumerate(seqs):
        rows = [_chunk_rows(tab, b, c, n, start) for c in range(C)]
        # dQ: per query chunk, per q head, contributions in step order.
        for cq in range(C):
            qrows, qpos = rows[cq]
            if len(qrows) == 0:
                continue
            for h in range(hq):
                g = kv_head_of(h, hq, hkv)
                acc = None
                for _, j in dq_contribution_order(cq, cp):
                    krows, kpos = rows[j]
                    if len(krows) == 0:
                        continue
                    c_dq, _, _ = masked_attention_backward(
                        q[qrows, h], k[krows, g], v[krows, g], do[qrows, h],
                        qpos, kpos, lse[qrows, h], delta[qrows, h], scale)
                    acc = c_dq if acc is None else acc + c_dq
                if acc is not None:
                    dq[qrows, h] = acc
        # dK/dV: per KV chunk, per kv head, contributions in ring order, the
        # first one used as the accumulator.
        for j in range(C):
            krows, kpos = rows[j]
            if len(krows) == 0:
                continue
            for g in range(hkv):
                acc_k = acc_v = None
                for _, _, cq in dkdv_contribution_order(j, cp):
                    qrows, qpos = rows[cq]
                    if len(qrows) == 0:
                        continue
                    for h in range(g * G, (g + 1) * G):
                        _, c_dk, c_dv = masked_attention_backward(
                            q[qrows, h], k[krows, g], v[krows, g], do[qrows, h],
                            qpos, kpos, lse[qrows, h], delta[qrows, h], scale)
                        if acc_k is None:
                            acc_k, acc_v = c_dk, c_dv
                        else:
                            acc_k = acc_k + c_dk
                            acc_v = acc_v + c_dv
                if acc_k is not None:
                    dk[krows, g] = acc_k
                    dv[krows, g] = acc_v
    return dq, dk, dv
