"""The allocation-free backward entry point, called through the C ABI.

ccg_attn_bwd_noalloc serves callers that cannot allocate device memory (a
plugin whose host framework owns all device memory, code that must not
call cudaMalloc once running): its scratch is a fixed array inside the
library.  It runs the same kernels as ccg_attn_bwd in the same fixed order,
so its gradients must be bitwise equal to those of ccg_attn_bwd (which takes
a caller-allocated workspace); the tests call it twice in a row, with and
without a caller status word, and compare bits.  A call whose sequence
offsets break the promise must leave the gradients unwritten and must not
poison the next call through the internal status word, and a problem too
large for the fixed scratch is rejected before anything is launched.
This file is collected last on purpose, and passes alone or after the rest.
"""

import ctypes

import pytest
import torch

from context_causal_gqa_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(lib, desc, x, o, lse, outs, status, cu_pad=None):
    L = lib.load()
    p = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    cpad = x["cu_seqlens_padded"] if cu_pad is None else cu_pad
    return L.ccg_attn_bwd_noalloc(ctypes.byref(desc), p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(x["do"]), p(lse),
                                  p(x["cu_seqlens"]), p(cpad), p(outs[0]), p(outs[1]),
                                  p(outs[2]), p(status),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _setup(lib, w):
    x = W.make_inputs(w, device="cuda")
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    ref = lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    desc = lib.make_desc(w.batch, w.hq, w.hkv, w.head_dim, w.cp, w.total_tokens)
    return x, o, lse, ref, desc


@pytest.mark.parametrize("w", [W.WORKLOADS["uniform"],
                               W.custom_workload("pad_d256", [700, 300], 4, 1, 256, 4, pad_to=64)],
                         ids=lambda w: w.name)
def test_noalloc_backward_bitwise_equals_regular_entry_point_twice(lib, w):
    x, o, lse, ref, desc = _setup(lib, w)
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in ref]
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if call == 0 else None
        code = _noalloc(lib, desc, x, o, lse, outs, status)
        assert code == 0, lib.status_str(code)
        torch.cuda.synchronize()
        if status is not None:
            assert lib.get_status(status) == 0
        for name, a, b in zip(("dQ", "dK", "dV"), outs, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name} (call {call}) differs from ccg_attn_bwd"


def test_noalloc_internal_status_word_is_cleared_by_every_call(lib):
    """With no caller status word, a call whose padded offsets break the
    promise (cu_seqlens_padded[B] != T) is detected on the device: the
    kernels skip their work and the gradients keep their previous contents.
    The next call clears the internal word and computes the gradients."""
    w = W.WORKLOADS["tiny"]
    x, o, lse, ref, desc = _setup(lib, w)
    bad = x["cu_seqlens_padded"].clone()
    bad[-1] += 2 * w.cp                                    # promise broken: last offset != T
    outs = [torch.full_like(t, float("nan")) for t in ref]
    code = _noalloc(lib, desc, x, o, lse, outs, None, cu_pad=bad)
    assert code == 0, lib.status_str(code)                 # not reported without a status word
    torch.cuda.synchronize()
    for t in outs:
        assert torch.isnan(t).all(), "a call with a broken promise must not write gradients"
    # the same broken call with a caller status word reports the device error
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = _noalloc(lib, desc, x, o, lse, outs, status, cu_pad=bad)
    assert code == 0
    assert lib.get_status(status) == 5                     # CCG_ERR_SEQLENS
    for t in outs:
        assert torch.isnan(t).all()
    # a valid call afterwards, again with no status word: the internal word
    # was cleared at its start, so the kernels run and match ccg_attn_bwd
    code = _noalloc(lib, desc, x, o, lse, outs, None)
    assert code == 0
    torch.cuda.synchronize()
    for name, a, b in zip(("dQ", "dK", "dV"), outs, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    desc = lib.make_desc(1, 32, 8, 128, 1, 1 << 20)     # Delta alone needs 128 MiB
    L = lib.load()
    null = ctypes.c_void_p(0)
    code = L.ccg_attn_bwd_noalloc(ctypes.byref(desc), *([null] * 12), null)
    assert code == 4, lib.status_str(code)               # CCG_ERR_WORKSPACE
