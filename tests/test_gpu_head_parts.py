"""Native head partitioning of the ring forward (ccg_attn_desc.head_parts;
TransformerEngine PR, Description and Native head partitioning: bounded
workspace): the ring-step partials and their LSE merge run over P head parts
in turn, reusing one set of partial slabs sized for Hq/P heads.  Every output
row gets the same partials merged in the same order as without partitioning,
so O and LSE must be bitwise equal to P = 1 -- on plain THD inputs, on
row-strided inputs (q, k, v sliced out of one fused buffer) and on the
head-split A2A layout -- and within tolerance of the FP64 oracle."""

import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_o_close, assert_lse_close

pytestmark = pytest.mark.gpu

CASES = [
    (W.custom_workload("hp_gqa4_d128_cp4_pad", [700, 300], 8, 2, 128, 4, pad_to=64), (2,)),
    (W.custom_workload("hp_gqa2_d256_cp2", [1024, 512], 8, 4, 256, 2), (2, 4)),
    (W.custom_workload("hp_mha_d128_cp8", [2048], 4, 4, 128, 8), (2, 4)),
]


def _bits_equal(a, b):
    return torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                       b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


@pytest.mark.parametrize("w,parts", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_head_parts_bitwise_equal_and_match_oracle(lib, w, parts):
    x = W.make_inputs(w, device="cuda")
    cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
    o1, l1 = lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp)
    for P in parts:
        desc1 = lib.make_desc(w.batch, w.hq, w.hkv, w.head_dim, w.cp, w.total_tokens)
        descP = lib.make_desc(w.batch, w.hq, w.hkv, w.head_dim, w.cp, w.total_tokens, head_parts=P)
        ws1, wsP = lib.workspace_size(desc1, 0), lib.workspace_size(descP, 0)
        assert wsP < ws1
        o = torch.full_like(o1, float("nan"))
        lse = torch.full_like(l1, float("nan"))
        lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp, out=o, lse=lse, head_parts=P)
        assert _bits_equal(o, o1), f"O with {P} head parts differs from the unpartitioned forward"
        assert _bits_equal(lse, l1), f"LSE with {P} head parts differs"
    o_ref, lse_ref = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.cu_seqlens,
                                              w.cu_seqlens_padded)
    assert_o_close(f64(o1), o_ref)
    assert_lse_close(f64(l1), lse_ref)


def test_head_parts_on_row_strided_inputs(lib):
    w = W.custom_workload("hp_pitch_d128_cp4", [700, 300], 8, 2, 128, 4, pad_to=8)
    x = W.make_inputs(w, device="cuda")
    T, hq, hkv, D = w.total_tokens, w.hq, w.hkv, w.head_dim
    qkv = torch.empty((T, hq + 2 * hkv, D), dtype=torch.bfloat16, device="cuda")
    qkv[:, :hq], qkv[:, hq:hq + hkv], qkv[:, hq + hkv:] = x["q"], x["k"], x["v"]
    q, k, v = qkv[:, :hq], qkv[:, hq:hq + hkv], qkv[:, hq + hkv:]
    cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
    o1, l1 = lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp)
    o2, l2 = lib.attn_fwd(q, k, v, cu, cpad, w.cp, head_parts=2)
    assert _bits_equal(o2, o1) and _bits_equal(l2, l1)


@pytest.mark.parametrize("P", [2, 4])
def test_head_parts_on_the_head_split_layout(lib, P):
    """In the head-split layout [G][T][H/G][D] a part is G/P whole head groups
    (one contiguous sub-tensor of q, k, v, o and lse)."""
    w = W.custom_workload("hp_split_d256_cp4", [1024, 512], 8, 4, 256, 4)
    x = W.make_inputs(w, device="cuda")
    cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
    qs, ks, vs = (lib.thd_pack(x[n], cpad, w.cp) for n in ("q", "k", "v"))
    o1, l1 = lib.attn_fwd(qs, ks, vs, cu, cpad, w.cp)
    oP, lP = lib.attn_fwd(qs, ks, vs, cu, cpad, w.cp, head_parts=P)
    assert _bits_equal(oP, o1) and _bits_equal(lP, l1)
