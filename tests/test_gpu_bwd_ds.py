"""The backward that keeps dS (a padded-length bound in the descriptor): the
dQ pass writes every unit's dS tile (at D = 256 its P tile too), the dK/dV
passes read them back (at D = 128 one dK/dV pass recomputing only P^T).  Checked against the FP64 oracle, against the
backward that recomputes them, for bitwise repeatability under NaN-poisoned
outputs, and for the device check of the bound.
"""

import numpy as np
import pytest
import torch

import oracle
from context_causal_gqa_gb300 import CCGError
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import assert_grad_close, f64, padding_rows

pytestmark = pytest.mark.gpu

SHAPES = [
    W.custom_workload("ds_gqa4_d256_cp2", [512], 4, 1, 256, 2),
    W.custom_workload("ds_gqa2_d256_cp4_pad", [300, 77], 4, 2, 256, 4, pad_to=64),
    W.custom_workload("ds_cp8_d256_pad", [700, 1500], 4, 1, 256, 8, pad_to=128),
    W.custom_workload("ds_mha_d256_cp2_pad", [384, 200], 2, 2, 256, 2, pad_to=64),
    W.custom_workload("ds_gqa8_d256_cp4_ragged", [1100, 36], 8, 1, 256, 4, pad_to=8),
    W.custom_workload("ds_empty_seqs_d256_cp2", [0, 300, 0, 77], 4, 2, 256, 2, pad_to=8),
    W.custom_workload("ds_cp16_d256_pad", [1000, 2100], 4, 1, 256, 16, pad_to=32),
    # several KV tiles a chunk: the dK/dV passes' CTA pairs (tiles 2i, 2i+1),
    # an odd last tile without a partner, ragged and padding tiles
    W.custom_workload("ds_gqa4_d256_cp2_t3", [1536, 1200], 4, 1, 256, 2, pad_to=128),
    W.custom_workload("ds_gqa2_d256_cp1_t4", [1024, 700, 260], 4, 2, 256, 1, pad_to=2),
]
MULTI_TILE = SHAPES[-2:]
SHAPES_D128 = [
    W.custom_workload("ds_gqa4_d128_cp2", [512], 4, 1, 128, 2),
    W.custom_workload("ds_gqa2_d128_cp4_pad", [300, 77], 4, 2, 128, 4, pad_to=64),
    W.custom_workload("ds_gqa8_d128_cp8_pad", [700, 1500], 8, 1, 128, 8, pad_to=128),
    W.custom_workload("ds_empty_seqs_d128_cp2", [0, 300, 0, 77], 4, 2, 128, 2, pad_to=8),
    W.custom_workload("ds_gqa4_d128_cp2_t3", [1536, 1200], 4, 1, 128, 2, pad_to=128),
    W.custom_workload("ds_gqa2_d128_cp1_t4", [1024, 700, 260], 4, 2, 128, 1, pad_to=2),
]


def _bound(w):
    return int(max(w.padded))


def _fwd(lib, x, w):
    return lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)


def _bwd(lib, x, w, o, lse, max_seqlen, **kw):
    return lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp,
                        max_seqlen=max_seqlen, **kw)


@pytest.mark.parametrize("w", SHAPES + SHAPES_D128, ids=lambda w: w.name)
def test_ds_backward_matches_oracle(lib, w):
    x = W.make_inputs(w, device="cuda")
    o, lse = _fwd(lib, x, w)
    dq, dk, dv = _bwd(lib, x, w, o, lse, _bound(w))
    ref = oracle.attention_backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), w.cu_seqlens,
                                    w.cu_seqlens_padded)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(f64(a), b, name)
    pad = padding_rows(w.cu_seqlens, w.cu_seqlens_padded)
    for a in (dq, dk, dv):
        assert np.all(f64(a)[pad] == 0)


@pytest.mark.parametrize("w", SHAPES[:3] + MULTI_TILE + SHAPES_D128[:1] + SHAPES_D128[-2:], ids=lambda w: w.name)
def test_ds_backward_agrees_with_the_recomputing_backward(lib, w):
    """Same dS and P values (the same arithmetic on the same S and dP, up to
    the tensor core's summation order in S versus S^T): dQ is that of the
    recomputing backward bit for bit (the same kernel), dK and dV agree to
    BF16 rounding."""
    x = W.make_inputs(w, device="cuda")
    o, lse = _fwd(lib, x, w)
    g0 = _bwd(lib, x, w, o, lse, 0)
    g1 = _bwd(lib, x, w, o, lse, _bound(w))
    assert torch.equal(g0[0], g1[0])
    for i in (1, 2):
        a, b = f64(g1[i]), f64(g0[i])
        assert np.linalg.norm(a - b) <= 1e-2 * np.linalg.norm(b) + 1e-6


@pytest.mark.parametrize("w", [SHAPES[2], SHAPES_D128[2]], ids=lambda w: w.name)
def test_ds_backward_bitwise_repeatable_under_poison(lib, w):
    x = W.make_inputs(w, device="cuda")
    o, lse = _fwd(lib, x, w)
    g1 = _bwd(lib, x, w, o, lse, _bound(w))
    for it in range(3):
        churn = [torch.empty(1 << (20 + it), device="cuda") for _ in range(4)]
        del churn
        outs = [torch.full_like(t, float("nan")) for t in g1]
        _bwd(lib, x, w, o, lse, _bound(w), dq=outs[0], dk=outs[1], dv=outs[2])
        for a, b in zip(outs, g1):
            assert torch.isfinite(a).all()
            assert torch.equal(a, b)


def test_ds_backward_larger_bound_same_bits(lib):
    """A looser bound only grows the dS region: the tiles' places and the
    result do not change."""
    w = SHAPES[1]
    x = W.make_inputs(w, device="cuda")
    o, lse = _fwd(lib, x, w)
    g1 = _bwd(lib, x, w, o, lse, _bound(w))
    g2 = _bwd(lib, x, w, o, lse, 4 * _bound(w))
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_ds_backward_broken_bound_is_reported_and_writes_nothing(lib):
    w = SHAPES[2]
    x = W.make_inputs(w, device="cuda")
    o, lse = _fwd(lib, x, w)
    outs = [torch.full_like(t, 7.0) for t in (x["q"], x["k"], x["v"])]
    with pytest.raises(CCGError) as e:
        _bwd(lib, x, w, o, lse, _bound(w) - 2 * w.cp, dq=outs[0], dk=outs[1], dv=outs[2])
    assert "SEQLENS" in str(e.value)
    for t in outs:
        assert torch.all(t == 7.0)


@pytest.mark.parametrize("D", [256, 128])
def test_ds_backward_head_split_layout_equals_plain(lib, D):
    """The head-split layout (head_groups = CP, the large workloads' A2A
    layout) gives the same gradients, bit for bit, as the plain layout."""
    w = W.custom_workload(f"ds_hs_d{D}", [2048, 1280], 8, 4, D, 4, pad_to=8)   # 2 KV tiles a chunk
    x = W.make_inputs(w, device="cuda")
    T, hg = w.total_tokens, w.cp
    o, lse = _fwd(lib, x, w)
    g1 = _bwd(lib, x, w, o, lse, _bound(w))

    def split(t):
        return t.view(T, hg, t.shape[1] // hg, t.shape[2]).transpose(0, 1).contiguous()

    def join(t, heads):
        return t.transpose(0, 1).reshape(T, heads, t.shape[3])

    q, k, v, do = (split(x[n]) for n in ("q", "k", "v", "do"))
    o2, lse2 = lib.attn_fwd(q, k, v, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, head_groups=hg)
    g2 = lib.attn_bwd(q, k, v, o2, do, lse2, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, head_groups=hg,
                      max_seqlen=_bound(w))
    for a, b, heads in zip(g1, g2, (w.hq, w.hkv, w.hkv)):
        assert torch.equal(a, join(b, heads))
