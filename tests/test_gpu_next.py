"""The next rows after the ring path: the forward with the merge folded into
one online softmax over all ring steps (ccg_attn_fwd_fused), and the A2A
(Ulysses-style) schedule end to end (pack -> full-sequence attention per
head group -> unpack), both against the FP64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from context_causal_gqa_gb300.pipeline import AttentionStep
from tests._gpu import f64, assert_o_close, assert_lse_close, assert_grad_close, padding_rows

pytestmark = pytest.mark.gpu

CASES = [
    W.WORKLOADS["tiny"],
    W.custom_workload("gqa3_d128_cp2", [384, 128], 3, 1, 128, 2),
    W.custom_workload("gqa2_d256_cp4_pad", [300, 77], 4, 2, 256, 4, pad_to=64),
    W.custom_workload("ragged_d128_cp4", [1000, 24, 1], 4, 2, 128, 4, pad_to=8),
    W.custom_workload("cp8_d256_pad", [700, 1500], 4, 1, 256, 8, pad_to=128),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_forward_matches_oracle(lib, w):
    x = W.make_inputs(w, device="cuda")
    o = torch.full_like(x["q"], float("nan"))
    lse = torch.full(x["q"].shape[:-1], float("nan"), device="cuda")
    lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, out=o, lse=lse, fused=True)
    o_ref, lse_ref = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.cu_seqlens,
                                              w.cu_seqlens_padded)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)
    assert np.all(f64(o)[padding_rows(w.cu_seqlens, w.cu_seqlens_padded)] == 0)
    # and the same (within rounding) as the ring-partials path
    o2, lse2 = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    assert float((o2.float() - o.float()).abs().max()) <= 2e-2


def test_fused_forward_full_size_d256_sampled(lib):
    w = W.WORKLOADS["d256"]
    x = W.make_inputs(w, device="cuda")
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, fused=True)
    G = w.hq // w.hkv
    for b, h in W.sample_pairs(w, 3):
        s0, n = int(w.cu_seqlens_padded[b]), w.seqlens[b]
        sl = slice(s0, s0 + n)
        o_ref, l_ref = oracle.head_forward(f64(x["q"][sl, h]), f64(x["k"][sl, h // G]), f64(x["v"][sl, h // G]))
        assert_o_close(f64(o[sl, h]), o_ref)
        assert np.max(np.abs(f64(lse[sl, h]) - l_ref)) <= 1e-3


@pytest.mark.parametrize("w", [W.custom_workload("a2a_d128", [512, 256], 8, 4, 128, 4),
                               W.custom_workload("a2a_d256_pad", [400, 130], 8, 2, 256, 2, pad_to=64)],
                         ids=lambda w: w.name)
def test_a2a_schedule_end_to_end(lib, w):
    x = W.make_inputs(w, device="cuda")            # read as the rank-major local layout
    step = AttentionStep(w, x, schedule="a2a")
    step.run()
    torch.cuda.synchronize()
    step.check()
    pi = torch.from_numpy(oracle.rank_major_token_index(w.cu_seqlens_padded, w.cp)).cuda()
    seq = {k: f64(x[k][pi]) for k in ("q", "k", "v", "do")}    # sequence-order tensors
    o_ref, _ = oracle.attention_forward(seq["q"], seq["k"], seq["v"], w.cu_seqlens, w.cu_seqlens_padded)
    g_ref = oracle.attention_backward(seq["q"], seq["k"], seq["v"], seq["do"], w.cu_seqlens, w.cu_seqlens_padded)
    assert_o_close(f64(step.o[pi]), o_ref)
    for name, a, r in zip(("dQ", "dK", "dV"), (step.dq, step.dk, step.dv), g_ref):
        assert_grad_close(f64(a[pi]), r, name)
