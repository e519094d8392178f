"""Backward parity: dQ pass (a6) and dK/dV pass (a7) through the C ABI vs the
FP64 oracle, plus bitwise repeatability under NaN-poisoned outputs,
allocator churn and changed-then-restored inputs."""

import numpy as np
import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_grad_close, padding_rows

pytestmark = pytest.mark.gpu

SMALL = [
    W.custom_workload("mha_d128_cp2", [256], 2, 2, 128, 2),
    W.custom_workload("gqa3_d128_cp2", [384, 128], 3, 1, 128, 2),
    W.custom_workload("gqa4_d256_cp2", [512], 4, 1, 256, 2),
    W.custom_workload("gqa2_d256_cp4_pad", [300, 77], 4, 2, 256, 4, pad_to=64),
    W.custom_workload("ragged_d128_cp4", [1000, 24, 1], 4, 2, 128, 4, pad_to=8),
    W.custom_workload("cp1_d128", [640], 4, 2, 128, 1),
    W.custom_workload("cp8_d128", [2048], 2, 1, 128, 8),
    W.custom_workload("cp8_d256_pad", [700, 1500], 4, 1, 256, 8, pad_to=128),
    W.custom_workload("mha_d256_cp2_pad", [384, 200], 2, 2, 256, 2, pad_to=64),
    W.custom_workload("gqa8_d256_cp4_ragged", [1100, 36], 8, 1, 256, 4, pad_to=8),
]


def _run(lib, x, w):
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    g = lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    return o, lse, g


def _check_full(lib, w):
    x = W.make_inputs(w, device="cuda")
    _, _, (dq, dk, dv) = _run(lib, x, w)
    ref = oracle.attention_backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), w.cu_seqlens,
                                    w.cu_seqlens_padded)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(f64(a), b, name)
    pad = padding_rows(w.cu_seqlens, w.cu_seqlens_padded)
    for a in (dq, dk, dv):
        assert np.all(f64(a)[pad] == 0)


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"]] + SMALL, ids=lambda w: w.name)
def test_backward_matches_oracle(lib, w):
    _check_full(lib, w)


def test_uniform_workload(lib):
    _check_full(lib, W.WORKLOADS["uniform"])


def test_unequal_workload_two_sequences(lib):
    w = W.WORKLOADS["unequal"]
    x = W.make_inputs(w, device="cuda")
    _, _, (dq, dk, dv) = _run(lib, x, w)
    rng = np.random.default_rng(w.seed)
    for b in rng.choice(w.batch, size=2, replace=False):
        s0, n, P = int(w.cu_seqlens_padded[b]), w.seqlens[b], w.padded[b]
        sl = slice(s0, s0 + n)
        ref = oracle.attention_backward(f64(x["q"][sl]), f64(x["k"][sl]), f64(x["v"][sl]), f64(x["do"][sl]),
                                        [0, n], [0, n])
        for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert_grad_close(f64(a[sl]), r, name)
            assert np.all(f64(a[s0 + n:s0 + P]) == 0)


def test_bitwise_repeatable_under_poison_churn_and_changed_inputs(lib):
    w = W.WORKLOADS["tiny"]
    x = W.make_inputs(w, device="cuda")
    o, lse, g1 = _run(lib, x, w)
    side = torch.cuda.Stream()
    for it in range(3):
        churn = [torch.empty(1 << (20 + it), device="cuda") for _ in range(4)]   # allocator churn
        del churn
        outs = [torch.full_like(t, float("nan")) for t in g1]
        with torch.cuda.stream(side):
            lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp,
                         dq=outs[0], dk=outs[1], dv=outs[2], stream=side)
        side.synchronize()
        for a, b in zip(outs, g1):
            assert torch.equal(a, b)
    # changed dO then restored: gradients change, then return to the same bits
    save = x["do"].clone()
    x["do"].mul_(0.5)
    g2 = lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    assert not torch.equal(g2[0], g1[0])
    x["do"].copy_(save)
    g3 = lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    for a, b in zip(g3, g1):
        assert torch.equal(a, b)


def test_first_contribution_is_the_accumulator(lib):
    """Outputs are written without any zero fill: poisoning dQ/dK/dV with NaN
    before the call must not leak into any element (every accumulator starts
    from its first contribution, padding rows are written as zeros)."""
    w = W.custom_workload("poison", [200, 56], 4, 2, 128, 4, pad_to=64)
    x = W.make_inputs(w, device="cuda")
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    dq = torch.full_like(x["q"], float("nan"))
    dk = torch.full_like(x["k"], float("nan"))
    dv = torch.full_like(x["v"], float("nan"))
    lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp,
                 dq=dq, dk=dk, dv=dv)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


# Chunk lengths are multiples of 128 and there is no padding: no query tile
# of the dK/dV pass reaches past its chunk.
@pytest.mark.parametrize("w", [W.custom_workload("zero_d128_cp4", [1024, 2048], 4, 2, 128, 4),
                               W.custom_workload("zero_d256_cp8", [2048], 4, 1, 256, 8)],
                         ids=lambda w: w.name)
def test_all_zero_contributions_give_exact_zeros(lib, w):
    """dO = -0.0 everywhere with q, k, v non-negative: every product that
    feeds dV (P * dO), dP (dO * V), dS and so dQ and dK is a zero, so every
    element of dQ, dK and dV, written over NaN, must come back as an exact
    zero.  The tensor core returns +0.0 for a sum of -0.0 products (measured
    on GB300: dV, a plain P^T dO product sum, comes back +0.0), so the sign
    of a zero cannot tell an accumulator that starts from its first
    contribution from one that starts from a zero fill; the zeros are checked
    bit for bit as +0.0."""
    x = W.make_inputs(w, device="cuda")
    for n in ("q", "k", "v"):
        x[n] = x[n].abs()
    x["do"] = torch.full_like(x["do"], -0.0)
    cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp)
    outs = [torch.full_like(x[n], float("nan")) for n in ("q", "k", "v")]
    lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, cu, cpad, w.cp, dq=outs[0], dk=outs[1], dv=outs[2])
    for name, g in zip(("dQ", "dK", "dV"), outs):
        bits = g.view(torch.int16)
        n_zero = int((bits == 0).sum())
        assert n_zero == bits.numel(), (f"{name}: {bits.numel() - n_zero} of {bits.numel()} elements are not +0.0 "
                                        f"(distinct bit patterns: {torch.unique(bits)[:8].tolist()})")
