"""Pins of the oracle's FP8 block-scaled expert functions against things other
than the oracle itself.

Source: atlasinference source page "spark_model/weight_loader/qwen3.rs",
load_layers (FP8 expert weights with one scale per 128 x 128 block, consumed
against wider activations, and a full-precision router option).  The code is
OCP E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
subnormals at a zero exponent field, no infinities, S.1111.111 NaN.

* ``fp8_e4m3_to_double``: the definition's special values, and every one of
  the 256 codes against torch's float8_e4m3fn conversion (a library routine).
* every finite E4M3 value is an fp16 value (the property that makes widening
  through fp16 exact).
* ``fp8_dequant_matrix``: a ragged matrix (neither side a multiple of 128, a
  non-square block grid, so a transposed scale index fails) against the
  library conversion times a scale grid expanded with ``np.repeat``.
* ``moe_ffn_fp8``: a dense brute force in numpy (library conversion, scipy
  ``expit``) with the ids and weights of the oracle router.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

torch = pytest.importorskip("torch")


def _lib_e4m3(codes) -> np.ndarray:
    """E4M3 codes -> float64 through torch's float8_e4m3fn dtype."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_special_values():
    v = oracle.fp8_e4m3_to_double
    assert v(0x00) == 0.0 and np.signbit(v(0x80)) and v(0x80) == 0.0
    assert v(0x38) == 1.0                       # exponent field 7 = bias
    assert v(0xB8) == -1.0
    assert v(0x40) == 2.0 and v(0xC0) == -2.0
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0   # largest finite
    assert v(0x08) == 2.0 ** -6                 # smallest normal
    assert v(0x01) == 2.0 ** -9                 # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert v(0x39) == 1.125                     # one mantissa step above 1
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    assert v(0x78) == 256.0                     # exponent field 15 is finite (no infinity)


def test_e4m3_all_codes_match_library():
    mine = np.array([oracle.fp8_e4m3_to_double(c) for c in range(256)])
    lib = _lib_e4m3(np.arange(256))
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2
    assert np.array_equal(mine[~nan], lib[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(lib[~nan]))


def test_e4m3_values_are_fp16_values():
    vals = np.array([oracle.fp8_e4m3_to_double(c) for c in range(256)])
    fin = vals[~np.isnan(vals)]
    assert np.array_equal(fin.astype(np.float16).astype(np.float64), fin)
    assert len(np.unique(fin)) == 253          # 254 finite codes, +0 and -0 equal


@pytest.mark.parametrize("rows,cols", [(200, 300), (128, 384), (1, 129)])
def test_dequant_matrix_ragged(rows, cols):
    codes, scales = synth.fp8_matrix(7, 99, 0, rows, cols, scale_base=0.25)
    assert scales.shape == (-(-rows // 128), -(-cols // 128))
    assert oracle.fp8_scale_count(rows, cols) == scales.size
    got = oracle.fp8_dequant_matrix(codes, scales, rows, cols)
    grid = np.repeat(np.repeat(scales.astype(np.float64), 128, axis=0), 128, axis=1)[:rows, :cols]
    want = _lib_e4m3(codes) * grid
    assert np.array_equal(got, want)


def test_dequant_matrix_one_hot_scale():
    # a single non-zero block scale lights exactly its 128 x 128 tile
    rows, cols = 256, 384
    codes = np.full((rows, cols), 0x38, dtype=np.uint8)        # every weight 1.0
    scales = np.zeros((2, 3), dtype=np.float32)
    scales[1, 2] = 3.0
    got = oracle.fp8_dequant_matrix(codes, scales, rows, cols)
    assert got[128:, 256:].min() == 3.0 and got[128:, 256:].max() == 3.0
    got[128:, 256:] = 0
    assert not got.any()


def test_dequant_rejects_size_mismatch():
    with pytest.raises(ValueError):
        oracle.fp8_dequant_matrix(np.zeros((4, 4), np.uint8), np.zeros(2, np.float32), 4, 4)


def _brute(inp, ids, w):
    x = inp["x"].astype(np.float64)
    H, F = inp["H"], inp["F"]

    def deq(codes, scales, rows, cols):
        grid = np.repeat(np.repeat(scales.astype(np.float64), 128, 0), 128, 1)[:rows, :cols]
        return _lib_e4m3(codes) * grid

    out = x.copy()
    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            e = ids[t, j]
            Wg = deq(inp["gate"][e], inp["gate_scale"][e], F, H)
            Wu = deq(inp["up"][e], inp["up_scale"][e], F, H)
            Wd = deq(inp["down"][e], inp["down_scale"][e], H, F)
            g, u = Wg @ x[t], Wu @ x[t]
            a = g * expit(g) * u
            out[t] += w[t, j] * (Wd @ a)
    return out


def test_moe_ffn_fp8_brute_force():
    inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS["tiny_fp8"])
    r = oracle.moe_forward_fp8(inp)
    want = _brute(inp, r["ids"], r["w"])
    assert np.abs(r["out"] - want).max() <= 1e-10 * np.abs(want).max()
    # the MoE term is of the order of x: a dropped term would show
    assert np.abs(r["out"] - inp["x"]).std() > 0.2


def test_moe_ffn_fp8_routing_is_the_f32_router():
    inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS["tiny_fp8"])
    r = oracle.moe_forward_fp8(inp)
    _, ids, w, _ = oracle.route(inp["x"], inp["router"], inp["K"])
    assert np.array_equal(r["ids"], ids) and np.array_equal(r["w"], w)


def test_moe_ffn_fp8_zero_scales_is_identity():
    inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS["tiny_fp8"])
    inp["down_scale"] = np.zeros_like(inp["down_scale"])
    r = oracle.moe_forward_fp8(inp)
    assert np.array_equal(r["out"], inp["x"].astype(np.float64))


def test_moe_ffn_fp8_rejects_bad_sizes():
    inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS["tiny_fp8"])
    with pytest.raises(ValueError):
        oracle.moe_ffn_fp8(inp["x"], np.zeros((inp["T"], inp["K"]), np.int32),
                           np.zeros((inp["T"], inp["K"])), inp["gate"], inp["gate_scale"][:-1],
                           inp["up"], inp["up_scale"], inp["down"], inp["down_scale"], inp["F"],
                           inp["E"])
