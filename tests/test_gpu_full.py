"""Full-size parity at the workloads' own sizes, in the launch configuration
bench.py times (the AttentionStep pipeline with the backward that keeps dS
and P), on seeded sampled
(sequence, q head) pairs the oracle computes one by one: O, LSE and dQ of
the sampled head, dK and dV of its kv head (the oracle sums its whole GQA
group).  Also checks that outputs are bitwise identical across three steps
written into NaN-poisoned outputs and poisoned workspaces, with
allocator churn in between, and that the A2A head-split
pack/unpack of the large workload is bit-exact at its full size (element
offsets past 2^31), against the oracle's index map."""

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


def _poison(step):
    """NaN into every output and intermediate the step writes, and 0xFF
    bytes (NaN patterns) over both workspaces (work plans, partials, Delta),
    with allocator churn: nothing may depend on what a previous run left."""
    churn = [torch.empty(1 << (20 + i), dtype=torch.uint8, device="cuda") for i in range(4)]
    for t in (step.o, step.dq, step.dk, step.dv, step.lse):
        t.fill_(float("nan"))
    if step.split:
        for t in (step.os, step.dqs, step.dks, step.dvs):
            t.fill_(float("nan"))
    for ws in (step.ws_f, step.ws_b):
        if ws.buf is not None:
            ws.buf.fill_(0xFF)
    del churn


@pytest.mark.parametrize("name", ["d256", "large"])
def test_full_size_sampled_pairs_and_repeatability(lib, name):
    from context_causal_gqa_gb300.pipeline import AttentionStep
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, device="cuda")
    step = AttentionStep(w, x, keep_ds=True)      # the bench's backward (keeps dS and P at D=256)
    assert step.max_seqlen > 0
    step.run()
    torch.cuda.synchronize()
    step.check()
    first = [t.clone() for t in (step.o, step.lse, step.dq, step.dk, step.dv)]
    for rep in range(2):                       # runs 2 and 3
        _poison(step)
        step.run()
        torch.cuda.synchronize()
        step.check()
        for nm, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), first, (step.o, step.lse, step.dq, step.dk, step.dv)):
            assert torch.equal(a.view(torch.int32 if a.dtype == torch.float32 else torch.int16),
                               b.view(torch.int32 if b.dtype == torch.float32 else torch.int16)), \
                f"{nm}: run {rep + 2} differs from run 1 (outputs must be bitwise identical)"
    del first
    _check_pairs(w, x, step, 4)
    del step, x
    torch.cuda.empty_cache()


def test_large_pack_unpack_bit_exact_at_full_size(lib):
    """A2A pack of q, k, v, dO of the large workload (q: 4.29e9 elements)
    against the oracle's rank-major index map on 4096+ seeded (head group,
    token) rows spread over the whole tensor, including rows whose element
    offsets exceed 2^31 (up to the last element, 2^32 - 1); unpack(pack(x)) == x
    on every element."""
    w = W.WORKLOADS["large"]
    assert w.pack_roundtrip
    x = W.make_inputs(w, device="cuda")
    T, cp = w.total_tokens, w.cp
    pi = oracle.rank_major_token_index(w.cu_seqlens_padded, cp)
    rng = np.random.default_rng(2024)
    n = 4096
    t_idx = rng.integers(0, T, size=n)
    g_idx = rng.integers(0, cp, size=n)
    edge_t = [0, 1, T // 2 - 1, T // 2, T - 2, T - 1]
    t_idx = np.concatenate([t_idx, np.repeat(edge_t, cp)])
    g_idx = np.concatenate([g_idx, np.tile(np.arange(cp), len(edge_t))])
    cpad = x["cu_seqlens_padded"]
    for name in ("q", "k", "v", "do"):
        src = x[name]
        H, D = src.shape[1], src.shape[2]
        hpg = H // cp
        packed = lib.thd_pack(src, cpad, cp)
        torch.cuda.synchronize()
        # for q and dO (4.29e9 elements) a quarter of the sampled rows start
        # past element 2^31 and the last one ends at element 2^32 - 1
        if H == w.hq:
            offs = ((g_idx.astype(np.int64) * T + t_idx) * hpg) * D
            assert offs.max() + hpg * D == src.numel() == (1 << 32) and (offs > (1 << 31)).sum() > n // 4
        tt = torch.from_numpy(t_idx).cuda()
        gg = torch.from_numpy(g_idx).cuda()
        got = packed[gg, tt]                                        # [N, H/cp, D]
        want = src.view(T, cp, hpg, D)[torch.from_numpy(pi[t_idx]).cuda(), gg]
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"{name}: packed rows differ from the index map"
        back = lib.thd_unpack(packed, cpad, cp)
        del packed
        assert torch.equal(back.view(torch.int16), src.view(torch.int16)), f"{name}: unpack(pack(x)) != x"
        del back
    del x
    torch.cuda.empty_cache()
