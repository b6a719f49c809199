"""qmoe_forward_noalloc: the allocation-free decode entry point.

It serves callers that cannot allocate device memory (their process's memory
belongs to another allocator, or allocation is forbidden in their hot loop).
These tests call it through the C ABI and check that two calls in a row give
the same result as the context-based qmoe_forward, within the fp32 tolerance
of the other parity tests, and that out-of-capacity sizes are refused.  The file
is collected last on purpose.
"""
import numpy as np
import pytest

import synth
from tests.compare import TOL_FP32, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import quantized_mixture_experts_f32_gb300 as q
    return q


@pytest.mark.parametrize("cfg_id", ["decode", "batch8", "tiny"])
def test_noalloc_matches_context_forward_twice(q, cfg_id):
    from tests import gpu_util as G
    inp = synth.moe_inputs(synth.MOE_CONFIGS[cfg_id])
    d = G.upload(inp)
    T, H, E, K, F = inp["T"], inp["H"], inp["E"], inp["K"], inp["F"]
    gt, ut, dt = q.QTYPE[inp["gate_t"]], q.QTYPE[inp["up_t"]], q.QTYPE[inp["down_t"]]
    stream = torch.cuda.current_stream(G.dev())
    ctx = G.make_ctx(q, inp)
    try:
        ref = torch.empty((T, H), dtype=torch.float32, device=G.dev())
        q.qmoe_forward(ctx, d["x"], d["router"], d["gate"], d["up"], d["down"], gt, ut, dt, T, ref)
        assert q.qmoe_get_status(ctx) == q.QMOE_OK
    finally:
        q.qmoe_destroy(ctx)
    for _ in range(2):
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device=G.dev())
        st = q.qmoe_forward_noalloc(d["x"], d["router"], d["gate"], d["up"], d["down"], gt, ut, dt,
                                    H, E, K, F, 1, T, out, stream.cuda_stream)
        assert st == q.QMOE_OK
        torch.cuda.synchronize()
        assert rel_err(out.cpu().numpy(), ref.cpu().numpy()) <= TOL_FP32


def test_noalloc_refuses_beyond_capacity(q):
    from tests import gpu_util as G
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"], T=9)
    d = G.upload(inp)
    out = torch.empty((9, inp["H"]), dtype=torch.float32, device=G.dev())
    st = q.qmoe_forward_noalloc(d["x"], d["router"], d["gate"], d["up"], d["down"], 1, 1, 1,
                                inp["H"], inp["E"], inp["K"], inp["F"], 1, 9, out, 0)
    assert st == 4                                    # QMOE_ERR_SHAPE, nothing enqueued
