"""The C ABI without a GPU: the library loads, exports every function that
include/ccg.h declares, and rejects bad arguments on the host before any CUDA
call (fail-closed error convention)."""

import ctypes
import os
import re

import pytest

import context_causal_gqa_gb300 as ccg
from context_causal_gqa_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ccg.h")


@pytest.fixture(scope="module")
def L():
    B.build()            # no-op when up to date; nvcc cross-compiles without a GPU
    return ccg.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ccg_\w+)\s*\(", text)))


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(B.LIB)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in ccg.h but not exported"
    # and the binding declares a prototype for each of them
    from context_causal_gqa_gb300._lib import SIGNATURES
    assert set(names) <= set(SIGNATURES), set(names) - set(SIGNATURES)


def test_status_strings(L):
    for code in range(8):
        assert len(ccg.status_str(code)) >= 2
    assert ccg.status_str(99) == "unknown status"


def _desc(**kw):
    d = dict(batch=1, hq=4, hkv=1, head_dim=128, cp=2, total_tokens=512)
    d.update(kw)
    return ccg.make_desc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), 2), (dict(head_dim=192), 2), (dict(hq=6, hkv=4), 2), (dict(cp=0), 2),
    (dict(cp=17), 2), (dict(total_tokens=510), 2), (dict(batch=0), 1), (dict(total_tokens=-4), 1),
])
def test_workspace_size_rejects_bad_descriptors(L, kw, code):
    assert ccg.workspace_size(_desc(**kw), False) == 0
    assert ccg.workspace_size(_desc(**kw), True) == 0


def test_row_pitch_validation_needs_no_gpu(L):
    dense = 4 * 128                                   # q row: Hq * D elements
    ok = _desc(pitches=(dense + 3 * 128, 1 * 128 + 8, 2 * 128, 0))       # e.g. a fused QKV buffer
    assert ccg.workspace_size(ok, False) > 0
    assert ccg.workspace_size(_desc(pitches=(dense, 128, 128, dense)), True) > 0   # explicit dense
    assert _call_fwd(L, _desc(pitches=(dense - 8, 0, 0, 0))) == 1       # pitch below H * D
    assert _call_fwd(L, _desc(pitches=(dense + 4, 0, 0, 0))) == 3       # not a multiple of 16 bytes
    assert _call_fwd(L, _desc(pitches=(0, 0, 0, 1004))) == 3            # dO pitch checked too
    assert _call_fwd(L, _desc(head_groups=2, hq=4, hkv=2, pitches=(1024, 0, 0, 0))) == 2   # head-split layout


def test_workspace_size_grows_with_problem(L):
    small, big = _desc(), _desc(total_tokens=4096)
    assert 0 < ccg.workspace_size(small, False) < ccg.workspace_size(big, False)
    # forward workspace holds CP partials of O (bf16) and LSE (fp32)
    assert ccg.workspace_size(big, False) >= 2 * 4096 * 4 * (128 * 2 + 4)
    assert ccg.workspace_size(big, True) >= 4096 * 4 * 4


def _call_fwd(L, desc, ptr=0x10000, ws=1 << 30, wsp=0x100000):
    p = ctypes.c_void_p(ptr)
    return L.ccg_attn_fwd(ctypes.byref(desc), p, p, p, p, p, p, p, ctypes.c_void_p(wsp), ws, p, None)


def test_host_side_rejections_need_no_gpu(L):
    assert L.ccg_attn_fwd(None, *([None] * 8), 0, None, None) == 1          # null descriptor
    assert _call_fwd(L, _desc(head_dim=64)) == 2                             # unsupported D
    assert _call_fwd(L, _desc(hq=5, hkv=2)) == 2                             # Hq % Hkv
    assert _call_fwd(L, _desc(), ptr=0x10008) == 3                           # misaligned tensor
    assert _call_fwd(L, _desc(), ws=16) == 4                                 # workspace too small
    assert _call_fwd(L, _desc(), wsp=0) == 4                                 # no workspace
    assert _call_fwd(L, _desc(), wsp=0x100010) == 3                          # workspace not 256-aligned
    null = ctypes.c_void_p(0)
    assert L.ccg_cp_lse_merge(0, None, None, 10, 128, null, null, None) == 1
    assert L.ccg_bwd_dot(null, null, 10, 128, null, None) == 1
    assert L.ccg_thd_pack(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), 1, 64, 6, 128, 4,
                          ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), None) == 2   # H % cp
    big = _desc(hq=32, hkv=8, total_tokens=1 << 20, cp=1)
    assert L.ccg_attn_bwd_noalloc(ctypes.byref(big), *([null] * 12), null) == 4
    # a padded-length bound adds the dS tiles to the workspace: a problem that
    # fits the allocation-free entry point's fixed scratch then exceeds it
    seq = _desc(hq=4, hkv=1, total_tokens=8192, cp=1)
    assert ccg.workspace_size(seq, True) < (1 << 24) - 256      # fits without the bound
    seq.max_seqlen = 8192
    assert ccg.workspace_size(seq, True) > (1 << 24)             # ~100 MB of dS tiles with it
    assert L.ccg_attn_bwd_noalloc(ctypes.byref(seq), *([null] * 12), null) == 4


def test_head_parts_shrink_the_forward_workspace_and_are_validated(L):
    import context_causal_gqa_gb300 as ccg
    T, hq, hkv, D, cp = 4096, 32, 8, 256, 8
    base = ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T), 0)
    partial_bytes = cp * T * hq * (D * 2 + 4)              # CP partial O (bf16) and LSE (float) slabs
    for P in (2, 4, 8):
        ws = ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_parts=P), 0)
        assert abs((base - ws) - partial_bytes * (1 - 1 / P)) <= 2 * 256
    # the backward and fused-forward workspaces hold no partials
    assert ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_parts=4), 1) == \
        ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T), 1)
    # whole GQA groups per part; whole head groups per part in the head-split layout
    assert ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_parts=3), 0) == 0
    assert ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_parts=16), 0) == 0
    assert ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_groups=2, head_parts=4), 0) == 0
    assert ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_groups=8, head_parts=4), 0) > 0
    assert ccg.workspace_size(ccg.make_desc(1, hq, hkv, D, cp, T, head_parts=-1), 0) == 0


def test_padded_length_bound_sizes_the_ds_backward_workspace(L):
    """max_seqlen > 0: the backward workspace adds one GQA group's dS tiles,
    and at D = 256 its P tiles too (t_max * (T / (128 * 2CP) + B) * CP(2CP+1)
    tiles of 32 KiB each per q head and kind, t_max = 128-row tiles of the
    longest chunk); with no bound it does not change, nor does the forward
    workspace; a negative bound is invalid."""
    import context_causal_gqa_gb300 as ccg
    B, T, hq, hkv, cp = 4, 4 * 8192, 32, 8, 8
    C = 2 * cp
    base = ccg.workspace_size(ccg.make_desc(B, hq, hkv, 256, cp, T), 1)
    ds = ccg.workspace_size(ccg.make_desc(B, hq, hkv, 256, cp, T, max_seqlen=8192), 1)
    t_max = -(-8192 // C // 128)
    tiles = t_max * (T // (128 * C) + B) * (C * (C + 1) // 2)
    extra = 2 * tiles * (hq // hkv) * 128 * 128 * 2 + (B + 1) * 8       # dS and P tiles
    assert 0 <= (ds - base) - extra <= 3 * 256
    base128 = ccg.workspace_size(ccg.make_desc(B, hq, hkv, 128, cp, T), 1)
    ds128 = ccg.workspace_size(ccg.make_desc(B, hq, hkv, 128, cp, T, max_seqlen=8192), 1)
    extra128 = tiles * (hq // hkv) * 128 * 128 * 2 + (B + 1) * 8          # dS tiles only
    assert 0 <= (ds128 - base128) - extra128 <= 3 * 256
    assert ccg.workspace_size(ccg.make_desc(B, hq, hkv, 256, cp, T, max_seqlen=8192), 0) == \
        ccg.workspace_size(ccg.make_desc(B, hq, hkv, 256, cp, T), 0)
    assert ccg.workspace_size(ccg.make_desc(B, hq, hkv, 256, cp, T, max_seqlen=-1), 1) == 0
