"""Forward parity: CUDA path (through the C ABI) vs the FP64 oracle.

Covers the ring-step partials (a3), the LSE merge inside the forward (a4),
D = 128 and 256, GQA groups of 1, 3, 4, padded unequal THD, the head-split
layout, repeatability and NaN-poisoned outputs.
"""

import numpy as np
import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import (f64, assert_o_close, assert_lse_close, padding_rows)

pytestmark = pytest.mark.gpu


def _inputs(w, seed=None):
    return W.make_inputs(w, device="cuda", seed=seed)


def _fwd(lib, x, w, head_groups=1):
    return lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp,
                        head_groups=head_groups)


def _oracle_fwd(x, w):
    return oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.cu_seqlens,
                                    w.cu_seqlens_padded)


SMALL = [
    W.custom_workload("mha_d128_cp2", [256], 2, 2, 128, 2),
    W.custom_workload("gqa3_d128_cp2", [384, 128], 3, 1, 128, 2),
    W.custom_workload("gqa4_d256_cp2", [512], 4, 1, 256, 2),
    W.custom_workload("gqa2_d256_cp4_pad", [300, 77], 4, 2, 256, 4, pad_to=64),
    W.custom_workload("ragged_d128_cp4", [1000, 24, 1], 4, 2, 128, 4, pad_to=8),
    W.custom_workload("cp1_d128", [640], 4, 2, 128, 1),
    W.custom_workload("cp8_d128", [2048], 2, 1, 128, 8),
    # D = 256, one q head per kv head: the single-CTA kernel (no head pairs)
    W.custom_workload("mha_d256_cp2", [384, 130], 2, 2, 256, 2, pad_to=4),
    # D = 256, groups of 4 over 2 kv heads: CTA pairs on (0,1), (2,3), ... of
    # each group, ragged sequences, every ring step of CP 8
    W.custom_workload("gqa4_d256_cp8_ragged", [2048, 700, 33], 8, 2, 256, 8, pad_to=16),
]


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"]] + SMALL, ids=lambda w: w.name)
def test_forward_matches_oracle(lib, w):
    x = _inputs(w)
    o, lse = _fwd(lib, x, w)
    o_ref, lse_ref = _oracle_fwd(x, w)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)
    pad = padding_rows(w.cu_seqlens, w.cu_seqlens_padded)
    assert np.all(f64(o)[pad] == 0)


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], SMALL[3], SMALL[6]], ids=lambda w: w.name)
def test_step_partials_match_oracle(lib, w):
    x = _inputs(w)
    parts = oracle.cp_forward_partials(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.cu_seqlens,
                                       w.cu_seqlens_padded, w.cp)
    for s in range(w.cp):
        o_p = torch.full_like(x["q"], float("nan"))
        l_p = torch.full(x["q"].shape[:-1], float("nan"), device="cuda")
        lib.attn_fwd_step(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, s, o_p, l_p)
        o_ref, l_ref = parts[s]
        present = np.isfinite(l_ref)
        og, lg = f64(o_p), f64(l_p)
        assert_o_close(og[present], o_ref[present], f"O_{s}")
        assert np.max(np.abs(lg[present] - l_ref[present])) <= 1e-3
        assert np.all(np.isnan(lg[~present])), "rows without a partial must be untouched"


def test_uniform_workload(lib):
    w = W.WORKLOADS["uniform"]
    x = _inputs(w)
    o, lse = _fwd(lib, x, w)
    o_ref, lse_ref = _oracle_fwd(x, w)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)


def test_unequal_workload_two_sequences(lib):
    w = W.WORKLOADS["unequal"]
    x = _inputs(w)
    o, lse = _fwd(lib, x, w)
    og, lg = f64(o), f64(lse)
    rng = np.random.default_rng(w.seed)
    for b in rng.choice(w.batch, size=2, replace=False):
        s0, n, P = int(w.cu_seqlens_padded[b]), w.seqlens[b], w.padded[b]
        sl = slice(s0, s0 + n)
        o_ref, l_ref = oracle.attention_forward(f64(x["q"][sl]), f64(x["k"][sl]), f64(x["v"][sl]),
                                                [0, n], [0, n])
        assert_o_close(og[sl], o_ref)
        assert_lse_close(lg[sl], l_ref)
        assert np.all(og[s0 + n:s0 + P] == 0) and np.all(np.isneginf(lg[s0 + n:s0 + P]))


def test_head_split_layout_equals_plain(lib):
    w = W.custom_workload("hs", [512, 256], 8, 4, 128, 4)
    x = _inputs(w)
    o, lse = _fwd(lib, x, w)
    T = w.total_tokens
    hg = w.cp
    def split(t):
        return t.view(T, hg, t.shape[1] // hg, t.shape[2]).transpose(0, 1).contiguous()
    o2, lse2 = lib.attn_fwd(split(x["q"]), split(x["k"]), split(x["v"]), x["cu_seqlens"],
                            x["cu_seqlens_padded"], w.cp, head_groups=hg)
    o2p = o2.transpose(0, 1).reshape(T, w.hq, w.head_dim)
    l2p = lse2.transpose(0, 1).reshape(T, w.hq)
    assert torch.equal(o2p, o), "head-split layout must give bit-identical results"
    assert torch.equal(l2p, lse)


def test_repeatable_and_poison_proof(lib):
    w = W.WORKLOADS["tiny"]
    x = _inputs(w)
    o1, l1 = _fwd(lib, x, w)
    o2 = torch.full_like(o1, float("nan"))
    l2 = torch.full_like(l1, float("nan"))
    lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, out=o2, lse=l2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # changed input then restored: same bits again
    q_save = x["q"].clone()
    x["q"].mul_(-1)
    o3, _ = _fwd(lib, x, w)
    assert not torch.equal(o3, o1)
    x["q"].copy_(q_save)
    o4, l4 = _fwd(lib, x, w)
    assert torch.equal(o4, o1) and torch.equal(l4, l1)
