"""Edge shapes against the FP64 oracle, forward (ring partials + merge, and
the fused forward) and backward: zero-length sequences, many short
sequences (most tiles ragged), and the largest emulated CP (16 ranks, 32
chunks per sequence)."""

import numpy as np
import pytest

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_o_close, assert_lse_close, assert_grad_close, padding_rows

pytestmark = pytest.mark.gpu

EDGES = [
    W.custom_workload("empty_seqs_d256_cp2", [0, 300, 0, 77], 4, 2, 256, 2, pad_to=8),
    W.custom_workload("empty_seqs_d128_cp4", [0, 0, 513, 0], 4, 1, 128, 4, pad_to=8),
    W.custom_workload("many_short_d128_cp2", [17] * 40 + [3], 4, 1, 128, 2, pad_to=4),
    W.custom_workload("cp16_d128", [4096], 2, 1, 128, 16),
    W.custom_workload("cp16_d256_pad", [1000, 2100], 4, 1, 256, 16, pad_to=32),
]


@pytest.mark.parametrize("w", EDGES, ids=lambda w: w.name)
def test_edge_forward_backward_match_oracle(lib, w):
    x = W.make_inputs(w, device="cuda")
    cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp)
    q, k, v, do = f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"])
    o_ref, lse_ref = oracle.attention_forward(q, k, v, w.cu_seqlens, w.cu_seqlens_padded)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)
    pad = padding_rows(w.cu_seqlens, w.cu_seqlens_padded)
    assert np.all(f64(o)[pad] == 0)
    # the fused forward over the same shapes
    of, lsef = lib.attn_fwd(x["q"], x["k"], x["v"], cu, cpad, w.cp, fused=True)
    assert_o_close(f64(of), o_ref, "O (fused)")
    assert_lse_close(f64(lsef), lse_ref)
    assert np.all(f64(of)[pad] == 0)
    dq, dk, dv = lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, cu, cpad, w.cp)
    ref = oracle.attention_backward(q, k, v, do, w.cu_seqlens, w.cu_seqlens_padded)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(f64(a), b, name)
        assert np.all(f64(a)[pad] == 0), f"{name}: padding rows not zero"
