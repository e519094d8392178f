"""Helpers shared by the GPU parity tests (comparison only, no attention math)."""

import numpy as np

# Tolerances (from the problem statement of the path): O, dQ, dK, dV relative
# L2 <= 1e-2; O max-abs <= 2e-2; LSE abs <= 1e-3 on real rows; padding rows
# exactly 0 / -inf; layout copies bit-exact.
REL_L2 = 1e-2
O_MAX_ABS = 2e-2
LSE_ABS = 1e-3


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_o_close(o_gpu, o_ref, what="O"):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite values"
    r = rel_l2(o_gpu, o_ref)
    m = float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0
    assert r <= REL_L2, f"{what}: rel-L2 {r:.3e} > {REL_L2}"
    assert m <= O_MAX_ABS, f"{what}: max-abs {m:.3e} > {O_MAX_ABS}"
    return r, m


def assert_grad_close(g_gpu, g_ref, what):
    assert np.all(np.isfinite(g_gpu)), f"{what}: non-finite values"
    r = rel_l2(g_gpu, g_ref)
    assert r <= REL_L2, f"{what}: rel-L2 {r:.3e} > {REL_L2}"
    return r


def assert_lse_close(l_gpu, l_ref, what="LSE"):
    fin = np.isfinite(l_ref)
    assert np.array_equal(fin, np.isfinite(l_gpu)), f"{what}: finite pattern differs"
    assert np.all(np.isneginf(l_gpu[~fin])), f"{what}: padding rows must be -inf"
    if fin.any():
        m = float(np.max(np.abs(l_gpu[fin] - l_ref[fin])))
        assert m <= LSE_ABS, f"{what}: max-abs {m:.3e} > {LSE_ABS}"


def padding_rows(cu, cu_pad):
    cu = np.asarray(cu)
    cu_pad = np.asarray(cu_pad)
    rows = [np.arange(cu_pad[b] + (cu[b + 1] - cu[b]), cu_pad[b + 1]) for b in range(len(cu) - 1)]
    return np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)
