"""Full-size parity at the workloads' own sizes, in the launch configuration
bench.py times (the AttentionStep pipeline), on seeded sampled
(sequence, q head) pairs the oracle computes one by one: O, LSE and dQ of
the sampled head, dK and dV of its kv head (the oracle sums its whole GQA
group).  Also checks that gradients are bitwise identical across two steps."""

import numpy as np
import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_o_close, assert_grad_close

pytestmark = pytest.mark.gpu


def _seq_rows(w, b, pi=None):
    s0, n = int(w.cu_seqlens_padded[b]), w.seqlens[b]
    rows = np.arange(s0, s0 + n)
    return rows if pi is None else pi[rows]


def _check_pairs(w, x, step, n_pairs):
    pi = oracle.rank_major_token_index(w.cu_seqlens_padded, w.cp) if w.pack_roundtrip else None
    G = w.hq // w.hkv
    for b, h in W.sample_pairs(w, n_pairs):
        rows = torch.from_numpy(_seq_rows(w, b, pi)).cuda()
        g = h // G
        kk, vv = f64(x["k"][rows, g]), f64(x["v"][rows, g])
        dk_ref = dv_ref = 0.0
        for hh in range(g * G, (g + 1) * G):
            dq, dk, dv, o, lse = oracle.head_backward(f64(x["q"][rows, hh]), kk, vv, f64(x["do"][rows, hh]))
            dk_ref = dk_ref + dk
            dv_ref = dv_ref + dv
            if hh == h:
                assert_o_close(f64(step.o[rows, h]), o, f"O seq{b} h{h}")
                assert_grad_close(f64(step.dq[rows, h]), dq, f"dQ seq{b} h{h}")
                if w.pack_roundtrip:
                    hpg = w.hq // w.cp
                    t = torch.from_numpy(_seq_rows(w, b)).cuda()
                    lse_gpu = f64(step.lse[h // hpg, t, h % hpg])
                else:
                    lse_gpu = f64(step.lse[rows, h])
                assert np.max(np.abs(lse_gpu - lse)) <= 1e-3, f"LSE seq{b} h{h}"
        assert_grad_close(f64(step.dk[rows, g]), dk_ref, f"dK seq{b} g{g}")
        assert_grad_close(f64(step.dv[rows, g]), dv_ref, f"dV seq{b} g{g}")


@pytest.mark.parametrize("name", ["d256", "large"])
def test_full_size_sampled_pairs_and_repeatability(lib, name):
    from context_causal_gqa_gb300.pipeline import AttentionStep
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, device="cuda")
    step = AttentionStep(w, x)
    step.run()
    torch.cuda.synchronize()
    step.check()
    first = [t.clone() for t in (step.o, step.dq, step.dk, step.dv)]
    step.run()
    torch.cuda.synchronize()
    for a, b in zip(first, (step.o, step.dq, step.dk, step.dv)):
        assert torch.equal(a, b), "outputs must be bitwise identical run to run"
    del first
    _check_pairs(w, x, step, 4)
    del step, x
    torch.cuda.empty_cache()
