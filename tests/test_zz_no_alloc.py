"""qmoe_forward_noalloc: the allocation-free decode entry point.

It serves callers that cannot allocate device memory: processes whose device
memory belongs to another allocator (a host framework's pool, a plugin loaded
into such a process), or loops in which a cudaMalloc, with its implicit device
synchronisation, must not happen after start-up.  These tests call it through
the C ABI, twice in a row, and check its output against the oracle and against
the context-based qmoe_forward, within the fp32 tolerance of the other parity
tests; they also check that shapes beyond its fixed scratch are refused before
anything is enqueued.  The file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle
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
def test_noalloc_matches_oracle_and_context_forward_twice(q, cfg_id):
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
    want = oracle.moe_forward(inp)["out"]
    for _ in range(2):
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device=G.dev())
        st = q.qmoe_forward_noalloc(d["x"], d["router"], d["gate"], d["up"], d["down"], gt, ut, dt,
                                    H, E, K, F, 1, T, out, stream.cuda_stream)
        assert st == q.QMOE_OK
        assert q.qmoe_noalloc_status(stream.cuda_stream) == q.QMOE_OK
        got = out.cpu().numpy()
        assert rel_err(got, want) <= TOL_FP32
        assert rel_err(got, ref.cpu().numpy()) <= TOL_FP32


def test_noalloc_refuses_beyond_capacity(q):
    from tests import gpu_util as G
    # more tokens than the fused decode kernel serves
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"], T=9)
    d = G.upload(inp)
    out = torch.empty((9, inp["H"]), dtype=torch.float32, device=G.dev())
    st = q.qmoe_forward_noalloc(d["x"], d["router"], d["gate"], d["up"], d["down"], 1, 1, 1,
                                inp["H"], inp["E"], inp["K"], inp["F"], 1, 9, out, 0)
    assert st == 4                                    # QMOE_ERR_SHAPE, nothing enqueued
    # a shape the fused kernel serves whose tagged buffers exceed the 2 MiB
    # scratch: 8 tokens at top-16 (the down outputs alone are 8*128*2048*8 B)
    inp16 = synth.moe_inputs(dict(synth.MOE_CONFIGS["batch8"], K=16))
    d16 = G.upload(inp16)
    ctx = G.make_ctx(q, inp16)
    try:
        assert q.qmoe_fused_decode_available(ctx, 8, 1, 1, 1)
    finally:
        q.qmoe_destroy(ctx)
    out16 = torch.full((8, inp16["H"]), 7.0, dtype=torch.float32, device=G.dev())
    st = q.qmoe_forward_noalloc(d16["x"], d16["router"], d16["gate"], d16["up"], d16["down"], 1, 1,
                                1, inp16["H"], inp16["E"], 16, inp16["F"], 1, 8, out16, 0)
    assert st == 4
    torch.cuda.synchronize()
    assert torch.all(out16 == 7.0)                    # nothing ran
