"""Parity of the CUDA MoE-FFN path with the CPU oracle, through the C ABI.

Workloads: the tiny config (H=256, E=8, k=2, F=256, T=4), the Qwen3-30B-A3B
layer at decode (T=1, Q6_K down), decode batch 8 (Q4_K down) and prefill
(T=512, biased router), plus ragged/edge cases.  Expert ids must match exactly
(up to F32 near-ties, see tests/compare.py), routing weights within 1e-5, and
outputs within max relative error 2e-3 on the fp32-accumulating decode path
(n_tokens <= 8) and 5e-3 on the half-precision tensor-core path (n_tokens > 8).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.compare import TOL_BF16, TOL_FP32, rel_err


def tol_for(T):
    return TOL_FP32 if T <= 8 else TOL_BF16

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


def _case(q, cfg_id, T=None, **over):
    cfg = dict(synth.MOE_CONFIGS[cfg_id], **over)
    inp = synth.moe_inputs(cfg, T=T)
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        got = G.run(q, ctx, inp, d)
    finally:
        q.qmoe_destroy(ctx)
    return inp, got


@pytest.mark.parametrize("cfg_id", ["tiny", "decode", "batch8"])
def test_decode_configs_match_oracle(q, cfg_id):
    inp, got = _case(q, cfg_id)
    err, ties, gap = G.check(inp, got, TOL_FP32, exact_ids=True)
    assert ties == []
    print(f"config {cfg_id}: rel err {err:.2e}, near-tie tokens {ties}, min k/k+1 gap {gap:.3e}")


def test_decode_sizes_take_the_fused_kernel(q):
    """Decode-size layers (T = 1 and T = 8 at the qwen3moe shape, both down
    qtypes) run as the single fused kernel; the T = 512 prefill does not."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    ctx = G.make_ctx(q, inp, max_tokens=512)
    try:
        for T in (1, 2, 4, 8):
            for dt in ("Q4_K", "Q6_K"):
                assert q.qmoe_fused_decode_available(ctx, T, q.QTYPE["Q4_K"], q.QTYPE["Q4_K"],
                                                     q.QTYPE[dt]), (T, dt)
        assert not q.qmoe_fused_decode_available(ctx, 9, q.QTYPE["Q4_K"], q.QTYPE["Q4_K"],
                                                 q.QTYPE["Q6_K"])
        assert not q.qmoe_fused_decode_available(ctx, 512, q.QTYPE["Q4_K"], q.QTYPE["Q4_K"],
                                                 q.QTYPE["Q6_K"])
    finally:
        q.qmoe_destroy(ctx)


def test_prefill_config_matches_oracle(q):
    inp, got = _case(q, "prefill")
    err, ties, gap = G.check(inp, got, TOL_BF16, exact_ids=True)
    assert ties == []
    counts = np.bincount(got["ids"].reshape(-1), minlength=inp["E"])
    assert counts.max() > 100 and (counts == 0).any()   # the bias skews routing
    print(f"prefill: rel err {err:.2e}, ties {ties}, gap {gap:.3e}, max/expert {counts.max()}")


@pytest.mark.parametrize("T", [2, 3, 7, 9, 33, 300])
def test_ragged_token_counts(q, T):
    inp, got = _case(q, "batch8", T=T)
    G.check(inp, got, tol_for(T))


@pytest.mark.parametrize("T,down_t", [(40, "Q6_K"), (21, "Q4_K"), (260, "Q6_K")])
def test_tensor_core_path_tiny_shapes(q, T, down_t):
    """n_tokens > 8 on the small geometry (one superblock per row): token tiles
    of 64/128/256 rows, ragged expert segments, both down formats."""
    inp, got = _case(q, "tiny", T=T, down_t=down_t)
    G.check(inp, got, TOL_BF16)


@pytest.mark.parametrize("gate_t,down_t", [("Q6_K", "Q4_K"), ("Q4_K", "Q4_K"), ("Q6_K", "Q6_K")])
def test_quant_type_combinations_tiny(q, gate_t, down_t):
    inp, got = _case(q, "tiny", gate_t=gate_t, up_t=gate_t, down_t=down_t)
    G.check(inp, got, TOL_FP32)


def test_top1_and_dense_topk(q):
    for K in (1, 8):
        inp, got = _case(q, "tiny", K=K)
        G.check(inp, got, TOL_FP32)
        if K == 8:
            assert all(sorted(r) == list(range(8)) for r in got["ids"].tolist())


def test_equal_logits_pick_lowest_indices(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    inp["router"] = np.zeros_like(inp["router"])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        got = G.run(q, ctx, inp, d)
    finally:
        q.qmoe_destroy(ctx)
    assert got["ids"].tolist() == [[0, 1]] * inp["T"]
    assert np.all(got["w"] == 0.5)
    G.check(inp, got, TOL_FP32)


def test_no_renorm_option(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp, norm=0)
    try:
        got = G.run(q, ctx, inp, d)
    finally:
        q.qmoe_destroy(ctx)
    G.check(inp, got, TOL_FP32, norm=False)


def test_residual_and_alias(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        res = np.random.default_rng(9).standard_normal((inp["T"], inp["H"])).astype(np.float32)
        rd = G.to_dev(res)
        got = G.run(q, ctx, inp, d, residual=rd, out=rd)          # out aliases residual
        G.check(inp, got, TOL_FP32, residual=res)
        xa = d["x"].clone()
        got2 = G.run(q, ctx, inp, d, x=xa, out=xa)                # out aliases input (decode)
        G.check(inp, got2, TOL_FP32)
    finally:
        q.qmoe_destroy(ctx)


def test_deterministic_and_batch_independent(q):
    """Repeated calls give bit-identical results; a token's result does not
    depend on the batch it is in: its ids are the same and its output agrees to
    fp32 rounding (a one-token call runs the batch-1 kernel, whose sums are
    associated differently from the batch kernel's)."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        a = G.run(q, ctx, inp, d)
        b = G.run(q, ctx, inp, d)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["ids"], b["ids"])
        for t in (0, 6):
            one = G.run(q, ctx, inp, d, T=1, x=d["x"][t:t + 1].contiguous())
            two = G.run(q, ctx, inp, d, T=1, x=d["x"][t:t + 1].contiguous())
            assert np.array_equal(one["out"], two["out"])
            assert np.array_equal(one["ids"][0], a["ids"][t])
            assert np.array_equal(one["w"][0], a["w"][t])
            assert rel_err(one["out"][0], a["out"][t]) <= 1e-6
    finally:
        q.qmoe_destroy(ctx)


def test_graph_capture_replays(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["decode"])
    d = G.upload(inp)
    out = torch.empty((1, inp["H"]), dtype=torch.float32, device=G.dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ctx = q.qmoe_create(q.make_config(inp["H"], inp["E"], inp["K"], inp["F"], 1, 1,
                                          s.cuda_stream))
        q.qmoe_forward(ctx, d["x"], d["router"], d["gate"], d["up"], d["down"], 1, 1, 2, 1, out)
        s.synchronize()
        ref = out.clone()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            q.qmoe_forward(ctx, d["x"], d["router"], d["gate"], d["up"], d["down"], 1, 1, 2, 1,
                           out)
        g.replay()
        s.synchronize()
    assert torch.equal(out, ref)
    q.qmoe_destroy(ctx)


def test_host_buffer_entry_point(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        hin = torch.from_numpy(inp["x"].copy()).pin_memory()
        hout = torch.empty_like(hin).pin_memory()
        q.qmoe_forward_host(ctx, hin, d["router"], d["gate"], d["up"], d["down"], 1, 1,
                            q.QTYPE[inp["down_t"]], inp["T"], hout)
        ref = oracle.moe_forward(inp)
        assert rel_err(hout.numpy(), ref["out"]) <= TOL_FP32
    finally:
        q.qmoe_destroy(ctx)


def test_argument_errors_are_reported_before_launch(q):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    out = torch.empty((inp["T"], inp["H"]), dtype=torch.float32, device=G.dev())
    try:
        cases = [
            (dict(n=inp["T"] + 1), 4),                        # n_tokens > max_tokens
            (dict(n=0), 4),
            (dict(gt=3), 3),                                   # unsupported qtype
            (dict(gate=d["gate"].view(-1)[1:]), 2),            # misaligned base
            (dict(gate=None), 1),                              # null pointer
        ]
        for over, status in cases:
            args = dict(n=inp["T"], gt=1, gate=d["gate"])
            args.update(over)
            with pytest.raises(q.QmoeError) as ei:
                q.qmoe_forward(ctx, d["x"], d["router"], args["gate"], d["up"], d["down"],
                               args["gt"], 1, 2, args["n"], out)
            assert ei.value.status == status, (over, ei.value)
        big = synth.moe_inputs(synth.MOE_CONFIGS["batch8"], T=9)
        bd = G.upload(big)
        c2 = G.make_ctx(q, big)
        try:
            with pytest.raises(q.QmoeError):
                q.qmoe_forward(c2, bd["x"], bd["router"], bd["gate"], bd["up"], bd["down"], 1, 1,
                               1, 9, bd["x"])                   # alias with T > 8
        finally:
            q.qmoe_destroy(c2)
        assert q.qmoe_get_status(ctx) == q.QMOE_OK
    finally:
        q.qmoe_destroy(ctx)


def test_guard_band_untouched(q):
    """Expert tensors placed between canary bytes: the canaries survive and the
    result is unchanged (no read or write outside the tensors' bytes matters)."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    d = G.upload(inp)
    pad = 4096
    bufs = {}
    for n in ("gate", "up", "down"):
        nb = inp[n].size
        buf = torch.full((nb + 2 * pad,), 0xA5, dtype=torch.uint8, device=G.dev())
        buf[pad:pad + nb] = d[n].view(-1)
        bufs[n] = buf
    dd = dict(d, **{n: bufs[n][pad:pad + inp[n].size] for n in bufs})
    ctx = G.make_ctx(q, inp)
    try:
        got = G.run(q, ctx, inp, dd)
    finally:
        q.qmoe_destroy(ctx)
    G.check(inp, got, TOL_FP32)
    for n, buf in bufs.items():
        assert torch.all(buf[:pad] == 0xA5) and torch.all(buf[-pad:] == 0xA5)


@pytest.mark.parametrize("T", [1, 8, 33])
def test_nan_token_stays_local(q, T):
    """A token whose activations are NaN gets NaN logits; ranking on order keys
    still yields a valid expert selection, so no kernel waits on a value that
    never comes (the status stays OK), and every other token is unaffected."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"], T=T)
    bad = T // 2
    inp["x"] = inp["x"].copy()
    inp["x"][bad, 5] = np.nan
    d = G.upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        got = G.run(q, ctx, inp, d)          # asserts QMOE_OK
    finally:
        q.qmoe_destroy(ctx)
    assert ((got["ids"] >= 0) & (got["ids"] < inp["E"])).all()
    assert not np.isfinite(got["out"][bad]).all()
    keep = [t for t in range(T) if t != bad]
    if keep:
        sub = dict(inp, T=len(keep), x=inp["x"][keep])
        ref = oracle.moe_forward(sub)
        tol = TOL_FP32 if T <= 8 else TOL_BF16
        assert rel_err(got["out"][keep], ref["out"]) <= tol


# ----------------------------------------------------------------------------- residual (A7)
# The weighted sum goes INTO the residual (aprender issue "qwen3moe ... has NO
# working CUDA path", "Gaps ... G3").  With the default inputs the MoE part is
# ~1e4 and the residual ~1, so a dropped or doubled residual would hide under
# the tolerance; these cases make the residual dominate or stand alone.
# Paths: fused decode (T = 1, 8), tensor-core prefill (T = 512), SIMT (Q6_K gate
# on the tiny shape), and the Q8_K-activation entry point.

RESIDUAL_CASES = [("decode", None, {}, TOL_FP32), ("batch8", None, {}, TOL_FP32),
                  ("prefill", None, {}, TOL_BF16),
                  ("tiny", None, {"gate_t": "Q6_K", "up_t": "Q6_K"}, TOL_FP32)]


@pytest.mark.parametrize("cfg_id,T,over,tol", RESIDUAL_CASES)
def test_large_residual_is_added_once(q, cfg_id, T, over, tol):
    """out = res + MoE(x) with res ~ 1e4 N(0,1): (out - res) must match the
    oracle's MoE part within the path's bound, so the residual is added exactly
    once and x is not used in its place."""
    inp = synth.moe_inputs(dict(synth.MOE_CONFIGS[cfg_id], **over), T=T)
    d = G.upload(inp)
    res = (1e4 * np.random.default_rng(11).standard_normal((inp["T"], inp["H"]))).astype(np.float32)
    ctx = G.make_ctx(q, inp)
    try:
        got = G.run(q, ctx, inp, d, residual=G.to_dev(res))
    finally:
        q.qmoe_destroy(ctx)
    ref = oracle.moe_forward(inp)
    assert np.array_equal(got["ids"], ref["ids"])
    moe_ref = ref["out"] - inp["x"].astype(np.float64)
    moe_got = got["out"].astype(np.float64) - res.astype(np.float64)
    err = rel_err(moe_got, moe_ref)
    assert err <= tol, f"MoE part (out - res) rel err {err:.3e} > {tol:.1e}"
    # a dropped residual, or x in its place, would miss by far more than the bound
    assert np.abs(res).max() > 100 * tol * np.abs(moe_ref).max()


@pytest.mark.parametrize("cfg_id,T,over,tol", RESIDUAL_CASES)
def test_zero_experts_return_the_residual_bit_for_bit(q, cfg_id, T, over, tol):
    """All-zero expert bytes dequantise to zero weights (d = dmin = 0), so every
    y_e is 0 and out must equal the residual exactly, bit for bit, while the
    routing still runs and matches the oracle."""
    inp = synth.moe_inputs(dict(synth.MOE_CONFIGS[cfg_id], **over), T=T)
    for n in ("gate", "up", "down"):
        inp[n] = np.zeros_like(inp[n])
    d = G.upload(inp)
    res = (1e4 * np.random.default_rng(12).standard_normal((inp["T"], inp["H"]))).astype(np.float32)
    ctx = G.make_ctx(q, inp)
    try:
        got = G.run(q, ctx, inp, d, residual=G.to_dev(res))
        got_x = G.run(q, ctx, inp, d)                  # residual = the input itself
    finally:
        q.qmoe_destroy(ctx)
    ref = oracle.moe_forward(inp)
    assert np.array_equal(got["ids"], ref["ids"])
    assert np.abs(got["w"] - ref["w"]).max() <= 1e-5
    assert np.array_equal(got["out"].view(np.uint32), res.view(np.uint32))
    assert np.array_equal(got_x["out"].view(np.uint32), inp["x"].view(np.uint32))
