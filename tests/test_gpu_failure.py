"""Failure paths, provoked on the host or by a wait that is made to run out.

Every cross-CTA wait of the fused decode kernel is bounded; on expiry the kernel
records QMOE_ERR_TIMEOUT in the context's status word, computes nothing more and
exits.  The test hook makes one launch wait for router logits that carry a
launch tag no CTA writes (a wait that cannot complete, with a 2 ms limit); the
status must say so, and the next normal call on the SAME context must match the
oracle, which shows that the launch tags and control words recover.  Nothing
here faults or hangs the GPU.

The workspace refusal states its arithmetic (bytes needed and free), as the
aprender issue "qwen3moe ... has NO working CUDA path" (later gap list) asks of
out-of-memory refusals: once through a real over-large configuration and once
through a hook that makes the allocation itself fail.
"""
import numpy as np
import pytest

import synth
from tests.compare import TOL_FP32

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


from tests import gpu_util as G  # noqa: E402


@pytest.mark.parametrize("cfg_id", ["decode", "batch8"])
def test_timed_out_wait_reports_and_the_context_recovers(q, cfg_id):
    inp = synth.moe_inputs(synth.MOE_CONFIGS[cfg_id])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        assert q.qmoe_fused_decode_available(ctx, inp["T"], 1, 1, q.QTYPE[inp["down_t"]])
        for _ in range(2):
            q.qmoe_debug_stall_next(ctx, 2_000_000)
            out = torch.zeros((inp["T"], inp["H"]), dtype=torch.float32, device=G.dev())
            q.qmoe_forward(ctx, d["x"], d["router"], d["gate"], d["up"], d["down"], 1, 1,
                           q.QTYPE[inp["down_t"]], inp["T"], out)
            assert q.qmoe_get_status(ctx) == 7                     # QMOE_ERR_TIMEOUT
            assert "status 7" in q.qmoe_last_error(ctx)
            assert q.qmoe_get_status(ctx) == q.QMOE_OK              # reading cleared it
            got = G.run(q, ctx, inp, d)                             # asserts QMOE_OK
            err, ties, _ = G.check(inp, got, TOL_FP32, exact_ids=True)
            assert ties == []
    finally:
        q.qmoe_destroy(ctx)


def test_stall_hook_rejects_zero_limit(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    ctx = G.make_ctx(q, inp)
    try:
        with pytest.raises(q.QmoeError):
            q.qmoe_debug_stall_next(ctx, 0)
    finally:
        q.qmoe_destroy(ctx)


def test_oversized_workspace_is_refused_with_its_arithmetic(q):
    # 2^20 tokens x top-16 x hidden 65536: the fp32 expert outputs alone are 4.4 TB
    cfg = q.make_config(65536, 1024, 16, 768, 1 << 20)
    need = q.qmoe_workspace_bytes(cfg)
    assert need > 4 * 10**12
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_create(cfg)
    assert ei.value.status == 5                                     # QMOE_ERR_NO_MEMORY
    msg = q.qmoe_last_error(None)
    assert f"needs {need} bytes" in msg and "free" in msg, msg


def test_failed_allocation_is_reported_and_the_next_create_works(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    q.qmoe_debug_fail_alloc(1)
    with pytest.raises(q.QmoeError) as ei:
        G.make_ctx(q, inp)
    assert ei.value.status == 5
    msg = q.qmoe_last_error(None)
    assert "bytes" in msg and "free" in msg, msg
    ctx = G.make_ctx(q, inp)                                        # the hook is spent
    try:
        got = G.run(q, ctx, inp, G.upload(inp))
        G.check(inp, got, TOL_FP32, exact_ids=True)
    finally:
        q.qmoe_destroy(ctx)
