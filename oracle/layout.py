"""A2A head-split pack / unpack index maps and the backward row dot, FP64 CPU.

Test infrastructure only (see the package docstring).  Shares nothing with
the CUDA path.

Sources (TransformerEngine PR "Optimize context parallel attention layouts
and gradient accumulation"):
  * Changes: a fast path for the A2A pack/unpack layout copies inside the
    existing swap API (Description, Changes).
  * Related optimization work / CP8 AllGather composition: the backward's row
    dot of O and dO over pitched rows, the per-row Delta = sum_d O*dO.

Reading of the A2A layouts (the pages name the copies but not the layout):
  * rank-major local layout [T, H, D]: for rank r = 0..CP-1, for sequence b:
    the rows of chunk r, then the rows of chunk 2CP-1-r (what each CP rank
    holds, concatenated over ranks);
  * head-split layout [CP, T, H/CP, D]: head group g holds heads
    g*H/CP .. (g+1)*H/CP-1 of ALL T tokens in sequence (physical THD) order;
  * pack:   out[g, t, h', :] = local[pi(t), g*H/CP + h', :]
    unpack: the inverse;  pi maps a sequence-order row to its rank-major row.
"""

import numpy as np

from .cp import chunk_table


def rank_major_token_index(cu_seqlens_padded, cp):
    """pi: sequence-order physical row -> rank-major row (int64 [T])."""
    tab = chunk_table(cu_seqlens_padded, cp)
    B, C, _ = tab.shape
    T = int(np.asarray(cu_seqlens_padded)[-1])
    order = []                      # rank-major list of sequence-order rows
    for r in range(cp):
        for b in range(B):
            for c in (r, C - 1 - r):
                c0, L = int(tab[b, c, 0]), int(tab[b, c, 1])
                order.append(np.arange(c0, c0 + L))
    order = np.concatenate(order) if order else np.zeros(0, dtype=np.int64)
    if len(order) != T:
        raise ValueError("cu_seqlens_padded does not cover T rows")
    pi = np.empty(T, dtype=np.int64)
    pi[order] = np.arange(T)
    return pi


def thd_pack(x_local, cu_seqlens_padded, cp):
    """Rank-major [T,H,D] -> head-split [CP,T,H/CP,D] (values copied exactly)."""
    x_local = np.asarray(x_local)
    T, H, D = x_local.shape
    if H % cp:
        raise ValueError("H must be a multiple of CP")
    hg = H // cp
    pi = rank_major_token_index(cu_seqlens_padded, cp)
    out = np.empty((cp, T, hg, D), dtype=x_local.dtype)
    for g in range(cp):
        out[g] = x_local[pi, g * hg:(g + 1) * hg, :]
    return out


def thd_unpack(x_split, cu_seqlens_padded, cp):
    """Head-split [CP,T,H/CP,D] -> rank-major [T,H,D]; inverse of thd_pack."""
    x_split = np.asarray(x_split)
    ncp, T, hg, D = x_split.shape
    if ncp != cp:
        raise ValueError("leading dimension must be CP")
    pi = rank_major_token_index(cu_seqlens_padded, cp)
    out = np.empty((T, cp * hg, D), dtype=x_split.dtype)
    for g in range(cp):
        out[pi, g * hg:(g + 1) * hg, :] = x_split[g]
    return out


def bwd_dot(o, do):
    """Delta[t, h] = sum_d O[t,h,d] * dO[t,h,d] in FP64."""
    return np.einsum("thd,thd->th", np.asarray(o, dtype=np.float64),
                     np.asarray(do, dtype=np.float64))
