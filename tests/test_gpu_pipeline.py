"""The host pipeline (AttentionStep.run_from_host_pipelined): steps whose
H2D/D2H copies overlap the neighbouring steps' compute on two device buffer
sets must return exactly what the plain step returns, for every step."""

import pytest
import torch

from context_causal_gqa_gb300 import workloads as W
from context_causal_gqa_gb300.pipeline import AttentionStep

pytestmark = pytest.mark.gpu

CASES = [
    W.WORKLOADS["tiny"],
    W.custom_workload("a2a_round_trip_d128_cp4", [640, 256], 8, 4, 128, 4, pad_to=8, pack_roundtrip=True),
    W.custom_workload("a2a_round_trip_d256_cp2", [512, 130], 4, 2, 256, 2, pad_to=4, pack_roundtrip=True),
]


@pytest.mark.parametrize("steps", [1, 2, 5])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_pipelined_host_steps_match_plain_step(lib, w, steps):
    x = W.make_inputs(w, device="cuda")
    step = AttentionStep(w, x)
    step.run()
    step.check()
    ref = [t.cpu() for t in step.output_tensors()]
    h_in, h_out = step.host_buffers()
    for d, h in zip(step.input_tensors(), h_in):
        h.copy_(d)
    for h in h_out:
        h.fill_(float("nan"))
    for t in step.output_tensors():          # the first set is overwritten by the pipeline too
        t.fill_(float("nan"))
    start, end = step.run_from_host_pipelined(h_in, h_out, steps)
    torch.cuda.synchronize()
    step.check()
    assert start.elapsed_time(end) > 0
    for name, a, r in zip(("o", "lse", "dq", "dk", "dv"), h_out, ref):
        assert torch.equal(a, r), f"{name}: pipelined host output differs from the plain step"
    # every buffer set that ran holds the same outputs
    for io in step.io[: min(steps, 2)]:
        for name, a, r in zip(("o", "lse", "dq", "dk", "dv"), io.outputs(), ref):
            assert torch.equal(a.cpu(), r), f"{name}: device buffer set differs"
