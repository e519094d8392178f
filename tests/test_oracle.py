"""Pins for the FP64 oracle: nothing here compares the oracle with itself.

Each test checks the oracle against something fixed outside it: a
hand-worked golden example, closed forms, brute-force scalar loops, a
library routine (torch CPU fp64 SDPA + autograd), finite differences, or a
structural identity of causal attention (masking, GQA = repeated-KV MHA,
chunked + LSE-merged = unchunked, padding invariance).  The last group
plants plausible mistakes in the oracle and checks that a pin catches each.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as oatt
from oracle import cp as ocp
from tests._brute import brute_forward, brute_backward

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------------------
# golden worked example (hand-derived)
# --------------------------------------------------------------------------

def test_golden_two_token_example():
    with open(os.path.join(GOLDEN, "two_token_worked_example.json")) as f:
        g = json.load(f)
    q, k, v, do = (np.array(g[x]) for x in ("q", "k", "v", "do"))
    o, lse = oatt.head_forward(q, k, v, g["scale"])
    assert np.allclose(o, g["o"], atol=1e-14, rtol=0)
    assert np.allclose(lse, g["lse"], atol=1e-14, rtol=0)
    dq, dk, dv, _, _ = oatt.head_backward(q, k, v, do, g["scale"])
    assert np.allclose(dq, g["dq"], atol=1e-14, rtol=0)
    assert np.allclose(dk, g["dk"], atol=1e-14, rtol=0)
    assert np.allclose(dv, g["dv"], atol=1e-14, rtol=0)
    # the same through the packed-THD entry points with a CP=1 split
    T = 2
    cu = np.array([0, 2])
    O, L = ocp.cp_attention_forward(q[:, None], k[:, None], v[:, None], cu, cu, 1, g["scale"])
    assert np.allclose(O[:, 0], g["o"], atol=1e-14) and np.allclose(L[:, 0], g["lse"], atol=1e-14)
    DQ, DK, DV = ocp.cp_attention_backward(q[:, None], k[:, None], v[:, None], do[:, None],
                                           cu, cu, 1, g["scale"])
    assert np.allclose(DQ[:, 0], g["dq"], atol=1e-14)
    assert np.allclose(DK[:, 0], g["dk"], atol=1e-14)
    assert np.allclose(DV[:, 0], g["dv"], atol=1e-14)
    assert T == 2


# --------------------------------------------------------------------------
# closed forms and invariants of the forward
# --------------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_causal_zeros():
    n, D = 24, 32                        # one-hot V: O rows are the P rows
    q = rnd((n, D), 1)
    k = rnd((n, D), 2)
    v = np.zeros((n, D))
    v[np.arange(n), np.arange(n)] = 1.0
    o, _ = oatt.head_forward(q, k, v)
    P = o[:, :n]
    assert np.max(np.abs(P.sum(axis=1) - 1.0)) <= 1e-13
    assert np.all(P[np.triu_indices(n, 1)] == 0.0)
    assert np.all(P[np.tril_indices(n)] > 0.0)


def test_causal_masking_is_exact():
    n, D, m = 40, 16, 17
    q, k, v = rnd((n, D), 3), rnd((n, D), 4), rnd((n, D), 5)
    o1, l1 = oatt.head_forward(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[m:] = rnd((n - m, D), 6) * 10
    v2[m:] = rnd((n - m, D), 7) * 10
    o2, l2 = oatt.head_forward(q, k2, v2)
    assert np.array_equal(o1[:m], o2[:m]) and np.array_equal(l1[:m], l2[:m])
    assert not np.allclose(o1[m:], o2[m:])


def test_closed_form_zero_queries_give_prefix_means():
    n, D = 33, 8
    v = rnd((n, D), 8)
    o, lse = oatt.head_forward(np.zeros((n, D)), rnd((n, D), 9), v)
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    assert np.max(np.abs(o - prefix_mean)) <= 1e-13
    assert np.max(np.abs(lse - np.log(np.arange(1, n + 1)))) <= 1e-13


def test_closed_form_first_row():
    n, D = 9, 16
    q, k, v = rnd((n, D), 10), rnd((n, D), 11), rnd((n, D), 12)
    o, lse = oatt.head_forward(q, k, v)
    assert np.array_equal(o[0], v[0])
    assert abs(lse[0] - np.dot(q[0], k[0]) / 4.0) <= 1e-14


def test_closed_form_single_token_gradients():
    D = 8
    q, k, v, do = (rnd((1, D), s) for s in (13, 14, 15, 16))
    dq, dk, dv, o, _ = oatt.head_backward(q, k, v, do)
    # dS = P (dP - Delta) with P = 1 and dP = Delta up to rounding of two dot orders
    assert np.max(np.abs(dq)) <= 1e-14 and np.max(np.abs(dk)) <= 1e-14
    assert np.array_equal(dv, do) and np.array_equal(o, v)


def test_scale_pin_uniform_keys():
    # all keys equal: P is uniform whatever the scale, and LSE = scale*<q,k> + ln(i+1)
    n, D = 12, 64
    q = rnd((n, D), 17)
    k = np.tile(rnd((1, D), 18), (n, 1))
    v = rnd((n, D), 19)
    _, lse = oatt.head_forward(q, k, v)
    expect = (q @ k[0]) / 8.0 + np.log(np.arange(1, n + 1))
    assert np.max(np.abs(lse - expect)) <= 1e-13


# --------------------------------------------------------------------------
# brute force, library cross-check, finite differences
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,hq,hkv,D", [(1, 2, 1, 4), (7, 4, 2, 8), (16, 4, 1, 8)])
def test_bruteforce_scalar_loops(n, hq, hkv, D):
    q, k, v, do = rnd((n, hq, D), 20), rnd((n, hkv, D), 21), rnd((n, hkv, D), 22), rnd((n, hq, D), 23)
    scale = 1.0 / math.sqrt(D)
    cu = np.array([0, n])
    O, L = oatt.attention_forward(q, k, v, cu)
    bo, bl = brute_forward(q.tolist(), k.tolist(), v.tolist(), scale)
    assert np.max(np.abs(O - np.array(bo))) <= 1e-12
    assert np.max(np.abs(L - np.array(bl))) <= 1e-12
    dq, dk, dv = oatt.attention_backward(q, k, v, do, cu)
    bq, bk, bv = brute_backward(q.tolist(), k.tolist(), v.tolist(), do.tolist(), scale)
    assert np.max(np.abs(dq - np.array(bq))) <= 1e-12
    assert np.max(np.abs(dk - np.array(bk))) <= 1e-12
    assert np.max(np.abs(dv - np.array(bv))) <= 1e-12


def test_library_crosscheck_torch_sdpa_fp64():
    torch = pytest.importorskip("torch")
    n, hq, hkv, D = 48, 8, 2, 32
    G = hq // hkv
    q, k, v, do = rnd((n, hq, D), 24), rnd((n, hkv, D), 25), rnd((n, hkv, D), 26), rnd((n, hq, D), 27)
    cu = np.array([0, n])
    O, L = oatt.attention_forward(q, k, v, cu)
    dq, dk, dv = oatt.attention_backward(q, k, v, do, cu)
    tq = torch.tensor(q.transpose(1, 0, 2), requires_grad=True)
    tk = torch.tensor(k.transpose(1, 0, 2), requires_grad=True)
    tv = torch.tensor(v.transpose(1, 0, 2), requires_grad=True)
    to = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, 0), tv.repeat_interleave(G, 0), is_causal=True)
    to.backward(torch.tensor(do.transpose(1, 0, 2)))
    assert np.max(np.abs(O - to.detach().numpy().transpose(1, 0, 2))) <= 1e-12
    assert np.max(np.abs(dq - tq.grad.numpy().transpose(1, 0, 2))) <= 1e-12
    assert np.max(np.abs(dk - tk.grad.numpy().transpose(1, 0, 2))) <= 1e-12
    assert np.max(np.abs(dv - tv.grad.numpy().transpose(1, 0, 2))) <= 1e-12
    # LSE against torch.logsumexp of the masked score matrix
    s = torch.einsum("hid,hjd->hij", tq.detach(), tk.detach().repeat_interleave(G, 0)) / math.sqrt(D)
    s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    assert np.max(np.abs(L - torch.logsumexp(s, -1).numpy().T)) <= 1e-12


def test_finite_differences_s32_prefix_of_tiny():
    """FD on the first 32 tokens of the tiny workload's shapes (Hq4/Hkv1, D128)."""
    n, hq, hkv, D = 32, 4, 1, 128
    q, k, v, do = rnd((n, hq, D), 28), rnd((n, hkv, D), 29), rnd((n, hkv, D), 30), rnd((n, hq, D), 31)
    cu = np.array([0, n])
    dq, dk, dv = oatt.attention_backward(q, k, v, do, cu)

    def loss(qq, kk, vv):
        O, _ = oatt.attention_forward(qq, kk, vv, cu)
        return float(np.sum(do * O))

    rng = np.random.default_rng(32)
    eps = 1e-6
    for name, grad, arr in (("q", dq, q), ("k", dk, k), ("v", dv, v)):
        scale = np.max(np.abs(grad))
        for _ in range(24):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            args = {"q": q, "k": k, "v": v}
            plus = {x: y.copy() for x, y in args.items()}
            minus = {x: y.copy() for x, y in args.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd = (loss(plus["q"], plus["k"], plus["v"]) - loss(minus["q"], minus["k"], minus["v"])) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, scale), (name, idx, fd, grad[idx])


# --------------------------------------------------------------------------
# structural identities
# --------------------------------------------------------------------------

def test_gqa_equals_repeated_kv_mha():
    n, hq, hkv, D = 30, 8, 2, 16
    G = hq // hkv
    q, k, v, do = rnd((n, hq, D), 33), rnd((n, hkv, D), 34), rnd((n, hkv, D), 35), rnd((n, hq, D), 36)
    cu = np.array([0, n])
    krep, vrep = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    O1, L1 = oatt.attention_forward(q, k, v, cu)
    O2, L2 = oatt.attention_forward(q, krep, vrep, cu)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    dq1, dk1, dv1 = oatt.attention_backward(q, k, v, do, cu)
    dq2, dk2, dv2 = oatt.attention_backward(q, krep, vrep, do, cu)
    assert np.array_equal(dq1, dq2)
    dk2s = dk2.reshape(n, hkv, G, D).sum(axis=2)
    dv2s = dv2.reshape(n, hkv, G, D).sum(axis=2)
    assert rel_err(dk1, dk2s) <= 1e-13 and rel_err(dv1, dv2s) <= 1e-13


def _thd_case(seqlens, padded, hq, hkv, D, seed):
    T = sum(padded)
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    cpad = np.concatenate([[0], np.cumsum(padded)])
    return (rnd((T, hq, D), seed), rnd((T, hkv, D), seed + 1), rnd((T, hkv, D), seed + 2),
            rnd((T, hq, D), seed + 3), cu, cpad)


@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_cp_chunked_merged_equals_unchunked(cp):
    seqlens = [64, 37, 80]
    padded = [64, 48, 96]            # multiples of 16 = 2*CP for every CP here
    q, k, v, do, cu, cpad = _thd_case(seqlens, padded, 4, 2, 16, 40 + cp)
    O1, L1 = oatt.attention_forward(q, k, v, cu, cpad)
    O2, L2 = ocp.cp_attention_forward(q, k, v, cu, cpad, cp)
    assert rel_err(O2, O1) <= 1e-12
    fin = np.isfinite(L1)
    assert np.array_equal(fin, np.isfinite(L2))
    assert np.max(np.abs(L2[fin] - L1[fin])) <= 1e-12
    g1 = oatt.attention_backward(q, k, v, do, cu, cpad)
    g2 = ocp.cp_attention_backward(q, k, v, do, cu, cpad, cp)
    for a, b in zip(g2, g1):
        assert rel_err(a, b) <= 1e-12


def test_padding_invariance_and_padding_outputs():
    seqlens, padded = [21, 40], [32, 48]
    q, k, v, do, cu, cpad = _thd_case(seqlens, padded, 4, 1, 8, 50)
    pad_rows = np.concatenate([np.arange(cpad[b] + seqlens[b], cpad[b + 1]) for b in range(2)])
    O1, L1 = ocp.cp_attention_forward(q, k, v, cu, cpad, 2)
    g1 = ocp.cp_attention_backward(q, k, v, do, cu, cpad, 2)
    for x in (q, k, v, do):
        x[pad_rows] = rnd(x[pad_rows].shape, 51) * 100
    O2, L2 = ocp.cp_attention_forward(q, k, v, cu, cpad, 2)
    g2 = ocp.cp_attention_backward(q, k, v, do, cu, cpad, 2)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)
    assert np.all(O1[pad_rows] == 0) and np.all(np.isneginf(L1[pad_rows]))
    for a in g1:
        assert np.all(a[pad_rows] == 0)


def test_lse_merge_special_cases():
    T, H, D = 5, 3, 4
    O = rnd((T, H, D), 60)
    L = rnd((T, H), 61)
    O1, L1 = ocp.lse_merge([(O, L)])
    assert np.array_equal(O1, O) and np.array_equal(L1, L)
    O2, L2 = ocp.lse_merge([(O, L), (3 * O, L)])
    assert np.allclose(O2, 2 * O, atol=1e-14) and np.allclose(L2, L + np.log(2), atol=1e-14)
    ninf = np.full((T, H), -np.inf)
    O3, L3 = ocp.lse_merge([(np.zeros_like(O), ninf), (O, L), (np.zeros_like(O), ninf)])
    assert np.array_equal(O3, O) and np.array_equal(L3, L)
    O4, L4 = ocp.lse_merge([(np.zeros_like(O), ninf)])
    assert np.all(O4 == 0) and np.all(np.isneginf(L4))
    # two partials over disjoint key sets of one row = attention over the union
    n, Dd = 10, 6
    qv, kv_, vv = rnd((1, Dd), 62), rnd((n, Dd), 63), rnd((n, Dd), 64)
    full_o, full_l = oatt.masked_attention(qv, kv_, vv, [n], np.arange(n), 0.3)
    a = oatt.masked_attention(qv, kv_[:4], vv[:4], [n], np.arange(4), 0.3)
    b = oatt.masked_attention(qv, kv_[4:], vv[4:], [n], np.arange(4, n), 0.3)
    mo, ml = ocp.lse_merge([(a[0][:, None], a[1][:, None]), (b[0][:, None], b[1][:, None])])
    assert np.allclose(mo[:, 0], full_o, atol=1e-14) and np.allclose(ml[:, 0], full_l, atol=1e-14)


# --------------------------------------------------------------------------
# the CP schedule itself
# --------------------------------------------------------------------------

@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_cp_schedule_covers_causal_pairs_once_and_balances(cp):
    C = 2 * cp
    seen = {}
    units = np.zeros((cp, cp))
    for s in range(cp):
        for r in range(cp):
            src = ocp.ring_source(r, s, cp)
            for cq in ocp.rank_chunks(r, cp):
                for j in ocp.visible_kv_chunks(cq, src, cp):
                    seen[(cq, j)] = seen.get((cq, j), 0) + 1
                    units[r, s] += 0.5 if j == cq else 1.0
    assert seen == {(c, j): 1 for c in range(C) for j in range(c + 1)}
    assert np.all(units == 2.0)          # every rank does 2 full-chunk units per step
    total = sum(len(ocp.partial_steps_for_chunk(c, cp)) for c in range(C))
    assert total == cp * cp + cp * (cp + 1) // 2
    for c in range(C):
        r = ocp.chunk_owner(c, cp)
        assert c in ocp.rank_chunks(r, cp)
        expect = list(range(cp)) if c >= cp else list(range(r + 1))
        assert ocp.partial_steps_for_chunk(c, cp) == expect
        order = ocp.dkdv_contribution_order(c, cp)
        assert order[0] == (0, r, c)                        # diagonal first
        assert sorted(x[2] for x in order) == list(range(c, C))
        assert [x[0] for x in order] == sorted(x[0] for x in order)
        dq = ocp.dq_contribution_order(c, cp)
        assert sorted(j for _, j in dq) == list(range(c + 1))
        assert dq[0][0] == 0 and [x[0] for x in dq] == sorted(x[0] for x in dq)
    if cp > 1:
        assert ocp.ring_source(1, 1, cp) == 0 and ocp.ring_source(0, 1, cp) == cp - 1


def test_chunk_table_and_padding_rule():
    tab = ocp.chunk_table([0, 64, 112], 2)
    assert tab.tolist() == [[[0, 16], [16, 16], [32, 16], [48, 16]],
                            [[64, 12], [76, 12], [88, 12], [100, 12]]]
    with pytest.raises(ValueError):
        ocp.chunk_table([0, 66], 2)


# --------------------------------------------------------------------------
# layout copies
# --------------------------------------------------------------------------

def _brute_pack(x, cpad, cp):
    C = 2 * cp
    T, H, D = x.shape
    hg = H // cp
    src_rows = []                         # rank-major order of sequence rows
    for r in range(cp):
        for b in range(len(cpad) - 1):
            L = (cpad[b + 1] - cpad[b]) // C
            for c in (r, C - 1 - r):
                for i in range(L):
                    src_rows.append(cpad[b] + c * L + i)
    out = np.zeros((cp, T, hg, D), dtype=x.dtype)
    for local_row, t in enumerate(src_rows):
        for g in range(cp):
            for hh in range(hg):
                out[g, t, hh] = x[local_row, g * hg + hh]
    return out


@pytest.mark.parametrize("cp", [1, 2, 4])
def test_pack_unpack_index_map(cp):
    cpad = np.array([0, 16, 48, 56])
    T, H, D = 56, 8, 3
    x = rnd((T, H, D), 70 + cp).astype(np.float32)
    p = oracle.thd_pack(x, cpad, cp)
    assert np.array_equal(p, _brute_pack(x, cpad, cp))
    assert np.array_equal(oracle.thd_unpack(p, cpad, cp), x)
    if cp == 1:
        assert np.array_equal(p[0], x)


def test_bwd_dot():
    o, do = rnd((6, 3, 5), 80), rnd((6, 3, 5), 81)
    d = oracle.bwd_dot(o, do)
    for t in range(6):
        for h in range(3):
            assert abs(d[t, h] - sum(o[t, h, i] * do[t, h, i] for i in range(5))) <= 1e-14


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# --------------------------------------------------------------------------

def _gqa_pin_holds():
    try:
        test_bruteforce_scalar_loops(7, 4, 2, 8)
        return True
    except AssertionError:
        return False


def test_planted_wrong_gqa_map_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "kv_head_of", lambda h, hq, hkv: h % hkv)
    assert not _gqa_pin_holds()


def test_planted_missing_scale_in_dq_is_caught(monkeypatch):
    real = oatt.masked_attention_backward

    def bad(Q, K, V, dO, qpos, kpos, lse, delta, scale):
        dQ, dK, dV = real(Q, K, V, dO, qpos, kpos, lse, delta, scale)
        return dQ / scale, dK, dV
    monkeypatch.setattr(oatt, "masked_attention_backward", bad)
    with pytest.raises(AssertionError):
        test_golden_two_token_example()


def test_planted_wrong_delta_sign_is_caught(monkeypatch):
    real = oatt.masked_attention_backward

    def bad(Q, K, V, dO, qpos, kpos, lse, delta, scale):
        return real(Q, K, V, dO, qpos, kpos, lse, -delta, scale)
    monkeypatch.setattr(oatt, "masked_attention_backward", bad)
    with pytest.raises(AssertionError):
        test_finite_differences_s32_prefix_of_tiny()


def test_planted_merge_without_rescale_is_caught(monkeypatch):
    def bad(parts):
        O = sum(np.asarray(p[0]) for p in parts)
        return O, np.max(np.stack([p[1] for p in parts]), axis=0)
    monkeypatch.setattr(ocp, "lse_merge", bad)
    with pytest.raises(AssertionError):
        test_cp_chunked_merged_equals_unchunked(2)


def test_planted_visible_future_chunk_is_caught(monkeypatch):
    monkeypatch.setattr(ocp, "visible_kv_chunks",
                        lambda cq, src, cp: list(ocp.rank_chunks(src, cp)))
    with pytest.raises(AssertionError):
        test_cp_schedule_covers_causal_pairs_once_and_balances(4)
