"""Parity of the CUDA MoE FFN over FP8 block-scaled experts (qmoe_forward_fp8)
with the oracle (oracle.moe_ffn_fp8), through the C ABI.

Source: atlasinference source page "spark_model/weight_loader/qwen3.rs",
load_layers (FP8 experts with one scale per 128 x 128 block; full-precision
router).  The kernels widen every E4M3 code exactly (through fp16) and sum in
fp32 against fp32 x and act, so the bound is the fp32 paths' one: max relative
error 2e-3.  Expert ids must match exactly up to F32 near-ties, weights within
1e-5.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.compare import TOL_BF16, TOL_FP32, TOL_W, ids_match, rel_err, tie_bound

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

NAMES = ("x", "router", "gate", "gate_scale", "up", "up_scale", "down", "down_scale")


def _upload(inp):
    return {n: G.to_dev(inp[n]) for n in NAMES}


def _call(q, ctx, d, T, K, out=None, x=None):
    H = d["x"].shape[1]
    x = d["x"] if x is None else x
    out = torch.empty((T, H), dtype=torch.float32, device=G.dev()) if out is None else out
    ids = torch.full((T, K), -1, dtype=torch.int32, device=G.dev())
    w = torch.full((T, K), -1.0, dtype=torch.float32, device=G.dev())
    q.qmoe_forward_fp8(ctx, x, d["router"], d["gate"], d["gate_scale"], d["up"], d["up_scale"],
                       d["down"], d["down_scale"], T, out, ids, w)
    assert q.qmoe_get_status(ctx) == q.QMOE_OK, q.qmoe_last_error(ctx)
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _check(inp, got, ids, w, exact_ids):
    logits, rids, rw, _ = oracle.route(inp["x"], inp["router"], inp["K"])
    ok, ties = ids_match(ids, rids, logits, tie_bound(logits))
    assert ok, f"expert ids differ beyond near-ties:\n{ids}\n{rids}"
    if exact_ids:
        assert ties == [], f"fixed-seed workload needed the near-tie allowance: {ties}"
    if ties:
        _, rids, rw, _ = oracle.route(inp["x"], inp["router"], inp["K"], force=ids)
    assert np.abs(w - rw).max() <= TOL_W
    want = oracle.moe_ffn_fp8(inp["x"], rids, rw, inp["gate"], inp["gate_scale"], inp["up"],
                              inp["up_scale"], inp["down"], inp["down_scale"], inp["F"], inp["E"])
    err = rel_err(got, want)
    tol = TOL_FP32 if inp["T"] <= GEMV_MAX else TOL_BF16
    assert err <= tol, f"max relative error {err:.3e} > {tol:.1e}"
    # the MoE term is not negligible against the residual
    assert np.abs(want - inp["x"]).max() > 0.1 * np.abs(inp["x"]).max()
    return err


GEMV_MAX = 32   # calls with more tokens run on the tensor cores (fp16 operands)

# (config, T, overrides): the tiny case spans several items per warp and a
# ragged token count; decode is the Qwen3-30B-A3B layer at T=1 and T=8 (the
# one-launch kernel) and T=16 (the multi-kernel GEMVs at that shape); T=32
# is the largest call on the CUDA-core GEMVs (two-launch routing), T=33 and
# T=40 the smallest on the tensor cores (token tiles shorter than 16 rows); the
# H=1024 / F=512 cases other unrolls and tile counts; T=512 the Qwen3-30B-A3B
# prefill shape (every expert hit, token tiles of up to 192 rows and ragged).
CASES = [
    ("tiny_fp8", None, {}),
    ("tiny_fp8", 1, {}),
    ("tiny_fp8", 32, {}),
    ("tiny_fp8", 33, {}),
    ("tiny_fp8", 40, {}),
    ("tiny_fp8", 7, {"H": 1024, "F": 512, "E": 16, "K": 4, "seed": 12}),
    ("tiny_fp8", 200, {"H": 1024, "F": 512, "E": 16, "K": 4, "seed": 12}),
    ("tiny_fp8", 3, {"E": 256, "K": 8, "seed": 30}),      # more than 128 experts: the generic top-k
    ("tiny_fp8", 40, {"E": 256, "K": 8, "seed": 30}),
    ("tiny_fp8", 4, {"E": 8, "K": 1, "seed": 31}),        # top-1
    ("decode_fp8", None, {}),
    ("decode_fp8", 8, {}),
    ("decode_fp8", 16, {}),
    ("decode_fp8", 512, {}),
]


@pytest.mark.parametrize("cfg_id,T,over", CASES)
def test_fp8_layer_matches_oracle(q, cfg_id, T, over):
    cfg = dict(synth.FP8_CONFIGS[cfg_id], **over)
    inp = synth.moe_inputs_fp8(cfg, T=T)
    d = _upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        got, ids, w = _call(q, ctx, d, inp["T"], inp["K"])
    finally:
        q.qmoe_destroy(ctx)
    err = _check(inp, got, ids, w, exact_ids=T is None)
    print(f"{cfg_id} T={inp['T']}: max relative error {err:.2e}")


# the GEMV path (tiny, T=6) and the one-kernel decode path (Qwen3 shape, T=1)
@pytest.mark.parametrize("cfg_id,T", [("tiny_fp8", 6), ("decode_fp8", 1)])
def test_fp8_in_place_and_repeatable(q, cfg_id, T):
    inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS[cfg_id], T=T)
    d = _upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        first, ids, w = _call(q, ctx, d, T, inp["K"])
        again, _, _ = _call(q, ctx, d, T, inp["K"])
        buf = d["x"].clone()
        inplace, _, _ = _call(q, ctx, d, T, inp["K"], out=buf, x=buf)
    finally:
        q.qmoe_destroy(ctx)
    assert np.array_equal(first, again), "two calls on the same inputs differ"
    assert np.array_equal(first, inplace), "hidden_out aliasing hidden_in changed the result"
    _check(inp, first, ids, w, exact_ids=True)


def test_fp8_rejects_bad_arguments(q):
    inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS["tiny_fp8"])
    d = _upload(inp)
    ctx = G.make_ctx(q, inp)
    out = torch.empty((inp["T"], inp["H"]), dtype=torch.float32, device=G.dev())
    try:
        with pytest.raises(RuntimeError, match="4-byte aligned"):
            q.qmoe_forward_fp8(ctx, d["x"], d["router"], d["gate"], d["gate_scale"].data_ptr() + 2,
                               d["up"], d["up_scale"], d["down"], d["down_scale"], inp["T"], out)
        with pytest.raises(RuntimeError, match="n_tokens"):
            q.qmoe_forward_fp8(ctx, d["x"], d["router"], d["gate"], d["gate_scale"], d["up"],
                               d["up_scale"], d["down"], d["down_scale"], inp["T"] + 1, out)
        with pytest.raises(RuntimeError, match="null"):
            q.qmoe_forward_fp8(ctx, d["x"], d["router"], d["gate"], None, d["up"],
                               d["up_scale"], d["down"], d["down_scale"], inp["T"], out)
    finally:
        q.qmoe_destroy(ctx)
