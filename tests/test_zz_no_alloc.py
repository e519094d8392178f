"""The allocation-free backward entry point, called through the C ABI.

ccg_attn_bwd_noalloc serves callers that cannot allocate device memory (a
plugin whose host framework owns all device memory, code that must not
call cudaMalloc once running): its scratch is a fixed array inside the
library.  These tests call it twice in a row and compare each result with
the regular ccg_attn_bwd (which takes a caller-allocated workspace), within
the gradient tolerance of the other tests, and check that a problem too
large for the fixed scratch is rejected before anything is launched.
This file is collected last on purpose, and passes alone or after the rest.
"""

import ctypes

import pytest
import torch

from context_causal_gqa_gb300 import workloads as W
from tests._gpu import f64, assert_grad_close

pytestmark = pytest.mark.gpu


def _noalloc(lib, desc, x, o, lse, outs, status):
    L = lib.load()
    p = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    return L.ccg_attn_bwd_noalloc(ctypes.byref(desc), p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(x["do"]), p(lse),
                                  p(x["cu_seqlens"]), p(x["cu_seqlens_padded"]), p(outs[0]), p(outs[1]),
                                  p(outs[2]), p(status),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("w", [W.WORKLOADS["uniform"],
                               W.custom_workload("pad_d256", [700, 300], 4, 1, 256, 4, pad_to=64)],
                         ids=lambda w: w.name)
def test_noalloc_backward_matches_regular_entry_point_twice(lib, w):
    x = W.make_inputs(w, device="cuda")
    o, lse = lib.attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    ref = lib.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, x["cu_seqlens"], x["cu_seqlens_padded"], w.cp)
    desc = lib.make_desc(w.batch, w.hq, w.hkv, w.head_dim, w.cp, w.total_tokens)
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in ref]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        code = _noalloc(lib, desc, x, o, lse, outs, status if call == 0 else None)
        assert code == 0, lib.status_str(code)
        torch.cuda.synchronize()
        assert lib.get_status(status) == 0
        for name, a, b in zip(("dQ", "dK", "dV"), outs, ref):
            assert_grad_close(f64(a), f64(b), f"{name} (call {call})")


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    desc = lib.make_desc(1, 32, 8, 128, 1, 1 << 20)     # Delta alone needs 128 MiB
    L = lib.load()
    null = ctypes.c_void_p(0)
    code = L.ccg_attn_bwd_noalloc(ctypes.byref(desc), *([null] * 12), null)
    assert code == 4, lib.status_str(code)               # CCG_ERR_WORKSPACE
