"""Parity of the HBM-bound steps: LSE merge (a4), Delta dot (a5), A2A
pack/unpack (a2, a8), the CP split table (a1) and the device promise check."""

import numpy as np
import pytest
import torch

import oracle
from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,D", [(1, 128), (3, 128), (8, 256), (16, 128)])
def test_lse_merge_matches_oracle(lib, K, D):
    g = torch.Generator(device="cuda").manual_seed(10 + K)
    rows = 1000
    o_parts = [torch.randn(rows, D, generator=g, device="cuda").bfloat16() for _ in range(K)]
    l_parts = [torch.randn(rows, generator=g, device="cuda") * 3 for _ in range(K)]
    # some partials absent
    for s in range(1, K, 2):
        l_parts[s][s::5] = float("-inf")
    l_parts[0][7] = float("-inf")
    if K == 1:
        l_parts[0][11] = float("-inf")
    o, lse = lib.cp_lse_merge(o_parts, l_parts)
    ref_o, ref_l = oracle.lse_merge([(f64(a), f64(b)) for a, b in zip(o_parts, l_parts)])
    assert_o_close(f64(o), ref_o)
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(f64(lse)))
    assert np.max(np.abs(f64(lse)[fin] - ref_l[fin])) <= 1e-5


@pytest.mark.parametrize("D", [128, 256])
def test_bwd_dot_matches_oracle(lib, D):
    g = torch.Generator(device="cuda").manual_seed(D)
    o = torch.randn(777, 3, D, generator=g, device="cuda").bfloat16()
    do = torch.randn(777, 3, D, generator=g, device="cuda").bfloat16()
    d = lib.bwd_dot(o, do)
    ref = oracle.bwd_dot(f64(o), f64(do))
    assert np.max(np.abs(f64(d) - ref)) <= 1e-4 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("cp,padded,H,D", [(1, [64, 32], 4, 128), (2, [64, 32, 128], 4, 128),
                                           (4, [64, 8 * 40, 8], 8, 256), (8, [16 * 5, 16 * 64], 32, 128)])
def test_pack_unpack_bit_exact(lib, cp, padded, H, D):
    cpad = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    T = int(cpad[-1])
    g = torch.Generator(device="cuda").manual_seed(cp)
    x = torch.randn(T, H, D, generator=g, device="cuda").bfloat16()
    cpad_t = torch.from_numpy(cpad).cuda()
    p = lib.thd_pack(x, cpad_t, cp)
    ref = oracle.thd_pack(x.view(torch.int16).cpu().numpy(), cpad, cp)
    assert np.array_equal(p.view(torch.int16).cpu().numpy(), ref)
    u = lib.thd_unpack(p, cpad_t, cp)
    assert torch.equal(u.view(torch.int16), x.view(torch.int16))


def test_cp_split_table(lib):
    w = W.WORKLOADS["unequal"]
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    cpad = torch.from_numpy(w.cu_seqlens_padded).cuda()
    tab = lib.cp_split(cu, cpad, w.cp, w.total_tokens)
    ref = oracle.chunk_table(w.cu_seqlens_padded, w.cp)
    assert np.array_equal(tab.cpu().numpy(), ref)


def test_broken_promise_sets_status_and_writes_nothing(lib):
    from context_causal_gqa_gb300 import CCGError
    w = W.WORKLOADS["tiny"]
    x = W.make_inputs(w, device="cuda")
    bad = torch.tensor([0, 510], dtype=torch.int32, device="cuda")       # 510 % 4 != 0
    cu = torch.tensor([0, 510], dtype=torch.int32, device="cuda")
    o = torch.full_like(x["q"], 7.0)
    lse = torch.full(x["q"].shape[:-1], 7.0, device="cuda")
    with pytest.raises(CCGError) as e:
        lib.attn_fwd(x["q"][:510], x["k"][:510], x["v"][:510], cu, bad, w.cp, out=o[:510], lse=lse[:510])
    assert "SEQLENS" in str(e.value) or "UNSUPPORTED" in str(e.value)
    # a promise that passes host checks but fails on device: S_b > P_b
    cu2 = torch.tensor([0, 600], dtype=torch.int32, device="cuda")
    cp2 = torch.tensor([0, 512], dtype=torch.int32, device="cuda")
    with pytest.raises(CCGError) as e:
        lib.attn_fwd(x["q"], x["k"], x["v"], cu2, cp2, w.cp, out=o, lse=lse)
    assert "SEQLENS" in str(e.value)
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)


def test_bounded_wait_times_out_into_status_and_context_stays_usable(lib):
    """Failure detection without a fault: a bounded wait that nothing
    satisfies gives up, the status word reports CCG_ERR_TIMEOUT, and the
    next computation on the same context is correct."""
    import ctypes
    L = lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = L.ccg_selftest_bounded_wait(ctypes.c_void_p(st.data_ptr()), 2000,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    assert lib.get_status(st) == 6                       # CCG_ERR_TIMEOUT
    assert L.ccg_selftest_bounded_wait(ctypes.c_void_p(st.data_ptr()), 0, None) == 1
    w = W.WORKLOADS["tiny"]
    x = W.make_inputs(w, device="cuda")
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    o_ref, _ = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.cu_seqlens, w.cu_seqlens_padded)
    assert_o_close(f64(o), o_ref)
