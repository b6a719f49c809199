"""Parity of the CUDA NVFP4 paths with the oracle, through the C ABI:
qmoe_forward_nvfp4 (the MoE layer over NVFP4 experts) against
oracle.moe_ffn_nvfp4, and qmoe_nvfp4_quantize (the BF16 -> NVFP4 runtime
quantiser) against oracle.nvfp4_quantize.

Source: atlasinference source page "spark_model/weight_loader/qwen3.rs",
load_layers (BF16 weights quantised to NVFP4 at load; a full-precision router
option).  The layer widens every E2M1 code and E4M3 scale exactly and sums in
fp32 against fp32 x and act, so its bound is the fp32 paths' one, max relative
error 2e-3; expert ids must match up to F32 near-ties, weights within 1e-5.  The
quantiser's codes, block scales and global scales are decided in fp32 on both
sides and must be bit-identical.
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

NAMES = ("x", "router", "gate", "gate_bs", "gate_gs", "up", "up_bs", "up_gs", "down", "down_bs",
         "down_gs")


def _upload(inp):
    return {n: G.to_dev(inp[n]) for n in NAMES}


def _call(q, ctx, d, T, K, out=None, x=None):
    H = d["x"].shape[1]
    x = d["x"] if x is None else x
    out = torch.empty((T, H), dtype=torch.float32, device=G.dev()) if out is None else out
    ids = torch.full((T, K), -1, dtype=torch.int32, device=G.dev())
    w = torch.full((T, K), -1.0, dtype=torch.float32, device=G.dev())
    q.qmoe_forward_nvfp4(ctx, x, d["router"], d["gate"], d["gate_bs"], d["gate_gs"], d["up"],
                         d["up_bs"], d["up_gs"], d["down"], d["down_bs"], d["down_gs"], T, out, ids,
                         w)
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
    want = oracle.moe_ffn_nvfp4(inp["x"], rids, rw, inp, inp["F"], inp["E"])
    err = rel_err(got, want)
    tol = TOL_FP32 if inp["T"] <= GEMV_MAX else TOL_BF16
    assert err <= tol, f"max relative error {err:.3e} > {tol:.1e}"
    assert np.abs(want - inp["x"]).max() > 0.1 * np.abs(inp["x"]).max()
    return err


GEMV_MAX = 32   # calls with more tokens run on the tensor cores (fp16 operands)

# tiny: several items per warp, ragged T; T=32 the largest GEMV call, T=33 and
# T=40 the smallest on the tensor cores; H=1024 / F=512 other unrolls and tile
# counts; decode: the Qwen3-30B-A3B layer at T=1 and 8 (the one-launch kernel),
# T=16 (the multi-kernel GEMVs at that shape); T=512 its prefill shape
CASES = [
    ("tiny_nvfp4", None, {}),
    ("tiny_nvfp4", 1, {}),
    ("tiny_nvfp4", 32, {}),
    ("tiny_nvfp4", 33, {}),
    ("tiny_nvfp4", 40, {}),
    ("tiny_nvfp4", 7, {"H": 1024, "F": 512, "E": 16, "K": 4, "seed": 22}),
    ("tiny_nvfp4", 200, {"H": 1024, "F": 512, "E": 16, "K": 4, "seed": 22}),
    ("tiny_nvfp4", 3, {"E": 256, "K": 8, "seed": 30}),      # more than 128 experts: the generic top-k
    ("tiny_nvfp4", 40, {"E": 256, "K": 8, "seed": 30}),
    ("tiny_nvfp4", 4, {"E": 8, "K": 1, "seed": 31}),        # top-1
    ("decode_nvfp4", None, {}),
    ("decode_nvfp4", 8, {}),
    ("decode_nvfp4", 16, {}),
    ("decode_nvfp4", 512, {}),
]


@pytest.mark.parametrize("cfg_id,T,over", CASES)
def test_nvfp4_layer_matches_oracle(q, cfg_id, T, over):
    cfg = dict(synth.NVFP4_CONFIGS[cfg_id], **over)
    inp = synth.moe_inputs_nvfp4(cfg, T=T)
    d = _upload(inp)
    ctx = G.make_ctx(q, inp)
    try:
        got, ids, w = _call(q, ctx, d, inp["T"], inp["K"])
    finally:
        q.qmoe_destroy(ctx)
    err = _check(inp, got, ids, w, exact_ids=T is None)
    print(f"{cfg_id} T={inp['T']}: max relative error {err:.2e}")


# the GEMV path (tiny, T=6) and the one-kernel decode path (Qwen3 shape, T=1)
@pytest.mark.parametrize("cfg_id,T", [("tiny_nvfp4", 6), ("decode_nvfp4", 1)])
def test_nvfp4_in_place_and_repeatable(q, cfg_id, T):
    inp = synth.moe_inputs_nvfp4(synth.NVFP4_CONFIGS[cfg_id], T=T)
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


@pytest.mark.parametrize("n_mats,rows,cols", [(3, 48, 96), (2, 768, 2048), (1, 5, 16)])
def test_quantize_bit_exact(q, n_mats, rows, cols):
    xs = [synth.bf16_matrix(40 + m, rows, cols) for m in range(n_mats)]
    if n_mats == 3:
        xs[1][:] = 0                                     # an all-zero matrix
        xs[2][0, :16] = np.uint16(0x8000)                # minus zeros in a block
    x = np.stack(xs)
    inp = dict(H=512, E=8, K=2, F=256, T=1)
    ctx = G.make_ctx(q, inp)
    try:
        xd = G.to_dev(x.view(np.int16))
        codes = torch.zeros((n_mats, rows, cols // 2), dtype=torch.uint8, device=G.dev())
        bs = torch.zeros((n_mats, rows, cols // 16), dtype=torch.uint8, device=G.dev())
        gl = torch.zeros(n_mats, dtype=torch.float32, device=G.dev())
        q.qmoe_nvfp4_quantize(ctx, xd, n_mats, rows, cols, codes, bs, gl)
        assert q.qmoe_get_status(ctx) == q.QMOE_OK, q.qmoe_last_error(ctx)
        codes, bs, gl = codes.cpu().numpy(), bs.cpu().numpy(), gl.cpu().numpy()
    finally:
        q.qmoe_destroy(ctx)
    for m in range(n_mats):
        wc, wb, wg = oracle.nvfp4_quantize(x[m])
        assert np.float32(gl[m]) == np.float32(wg), (m, gl[m], wg)
        assert np.array_equal(bs[m], wb), f"matrix {m}: block scales differ"
        assert np.array_equal(codes[m], wc), f"matrix {m}: codes differ"


def test_nvfp4_rejects_bad_arguments(q):
    inp = synth.moe_inputs_nvfp4(synth.NVFP4_CONFIGS["tiny_nvfp4"])
    d = _upload(inp)
    ctx = G.make_ctx(q, inp)
    out = torch.empty((inp["T"], inp["H"]), dtype=torch.float32, device=G.dev())
    args = [d[n] for n in NAMES[1:]]
    try:
        bad = list(args)
        bad[2] = d["gate_bs"].data_ptr() + 1                  # odd block-scale pointer
        with pytest.raises(RuntimeError, match="2-byte aligned"):
            q.qmoe_forward_nvfp4(ctx, d["x"], *bad, inp["T"], out)
        with pytest.raises(RuntimeError, match="n_tokens"):
            q.qmoe_forward_nvfp4(ctx, d["x"], *args, inp["T"] + 1, out)
        with pytest.raises(RuntimeError, match="multiple of 16"):
            q.qmoe_nvfp4_quantize(ctx, d["x"], 1, 4, 24, d["gate"], d["gate_bs"], d["gate_gs"])
    finally:
        q.qmoe_destroy(ctx)
