"""Physical-pitch (row-strided) THD inputs: q, k, v sliced out of one fused
[T][Hq+2Hkv][D] projection buffer, and dO a slice of a wider buffer, must
give exactly what the same values give when copied dense (the kernels read
the same numbers through their tensor maps), for the ring forward, the
fused forward and the backward; and both must match the FP64 oracle."""

import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_o_close, assert_grad_close

pytestmark = pytest.mark.gpu

CASES = [
    W.custom_workload("pitch_gqa4_d128_cp4", [700, 300], 8, 2, 128, 4, pad_to=8),
    W.custom_workload("pitch_gqa2_d256_cp2", [512, 77], 4, 2, 256, 2, pad_to=4),
]


def _strided(x, w):
    T, hq, hkv, D = w.total_tokens, w.hq, w.hkv, w.head_dim
    qkv = torch.empty((T, hq + 2 * hkv, D), dtype=torch.bfloat16, device="cuda")
    qkv[:, :hq] = x["q"]
    qkv[:, hq:hq + hkv] = x["k"]
    qkv[:, hq + hkv:] = x["v"]
    wide = torch.full((T, hq + 3, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    wide[:, 1:hq + 1] = x["do"]
    q, k, v, do = qkv[:, :hq], qkv[:, hq:hq + hkv], qkv[:, hq + hkv:], wide[:, 1:hq + 1]
    assert not q.is_contiguous() and q.stride(0) == (hq + 2 * hkv) * D and do.stride(0) == (hq + 3) * D
    return q, k, v, do


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_row_strided_inputs_match_dense(lib, w):
    x = W.make_inputs(w, device="cuda")
    cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
    q, k, v, do = _strided(x, w)
    for fused in (False, True):
        o_d, lse_d = lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp, fused=fused)
        o_s, lse_s = lib.attn_fwd(q, k, v, cu, cpad, w.cp, fused=fused)
        assert torch.equal(o_s, o_d) and torch.equal(lse_s, lse_d), f"forward (fused={fused})"
    g_d = lib.attn_bwd(x["q"], x["k"], x["v"], o_d, x["do"], lse_d, cu, cpad, w.cp)
    g_s = lib.attn_bwd(q, k, v, o_d, do, lse_d, cu, cpad, w.cp)
    for name, a, b in zip(("dQ", "dK", "dV"), g_s, g_d):
        assert torch.equal(a, b), f"{name}: strided inputs differ from dense"
    o_ref, _ = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.cu_seqlens, w.cu_seqlens_padded)
    assert_o_close(f64(o_s), o_ref)
    ref = oracle.attention_backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), w.cu_seqlens,
                                    w.cu_seqlens_padded)
    for name, a, b in zip(("dQ", "dK", "dV"), g_s, ref):
        assert_grad_close(f64(a), b, name)


def test_strided_outputs_are_rejected(lib):
    w = CASES[0]
    x = W.make_inputs(w, device="cuda")
    wide = torch.empty((w.total_tokens, w.hq + 1, w.head_dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp, out=wide[:, :w.hq])
