"""Pins of the oracle's NVFP4 functions against things other than the oracle.

Source: atlasinference source page "spark_model/weight_loader/qwen3.rs",
load_layers (dense weights quantised from BF16 to NVFP4 at load by a global
absmax pass and a quantisation pass).  NVFP4 is the public format: FP4 E2M1
elements (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; magnitudes 0,
0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per 16 consecutive elements and one
fp32 scale per tensor.

* ``e2m1_to_double``: the format's value table.
* ``nvfp4_dequant_matrix``: a numpy brute force (table lookup, torch's E4M3
  conversion), with nibble order and the scale index exercised by one-hot cases.
* ``moe_ffn_nvfp4``: a dense numpy brute force with the oracle router's ids.
* ``nvfp4_quantize``: every decision checked by brute-force optimality: the
  global scale is amax / 2688, each block scale is the E4M3 value nearest to
  bmax / (6 global) (ties to the even code), each code the E2M1 value nearest to
  x / d (ties to the even code, saturating at 6); an exactly representable
  matrix comes back exactly; the round trip is within half a step.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

torch = pytest.importorskip("torch")

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]    # the format's magnitudes by code


def _e4m3(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _bf16(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _deq(codes, bs, g, rows, cols):
    lo, hi = codes & 15, codes >> 4
    q = np.empty((rows, cols), dtype=np.uint8)
    q[:, 0::2], q[:, 1::2] = lo, hi
    tab = np.array(E2M1 + [-v for v in E2M1])
    return tab[q] * np.repeat(_e4m3(bs), 16, axis=1) * np.float64(g)


def test_e2m1_table():
    for c in range(8):
        assert oracle.e2m1_to_double(c) == E2M1[c]
        v = oracle.e2m1_to_double(c | 8)
        assert v == -E2M1[c] and np.signbit(v)


def test_dequant_matches_brute_force():
    codes, bs, g = synth.nvfp4_matrix(3, 99, 0, 48, 96)
    got = oracle.nvfp4_dequant_matrix(codes, bs, g, 48, 96)
    assert np.array_equal(got, _deq(codes, bs, g, 48, 96))


def test_dequant_nibble_order_and_scale_index():
    rows, cols = 2, 64
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    codes[1, 9] = 0x70            # element 19 of row 1 (high nibble of byte 9) = 6.0
    bs = np.full((rows, cols // 16), 0x38, dtype=np.uint8)   # all block scales 1.0
    bs[1, 1] = 0x40               # elements 16..31 of row 1: scale 2.0
    got = oracle.nvfp4_dequant_matrix(codes, bs, 0.5, rows, cols)
    want = np.zeros((rows, cols))
    want[1, 19] = 6.0 * 2.0 * 0.5
    assert np.array_equal(got, want)


def test_moe_ffn_nvfp4_brute_force():
    inp = synth.moe_inputs_nvfp4(synth.NVFP4_CONFIGS["tiny_nvfp4"])
    r = oracle.moe_forward_nvfp4(inp)
    x = inp["x"].astype(np.float64)
    H, F = inp["H"], inp["F"]
    want = x.copy()
    for t in range(inp["T"]):
        for j in range(inp["K"]):
            e = r["ids"][t, j]
            Wg = _deq(inp["gate"][e], inp["gate_bs"][e], inp["gate_gs"][e], F, H)
            Wu = _deq(inp["up"][e], inp["up_bs"][e], inp["up_gs"][e], F, H)
            Wd = _deq(inp["down"][e], inp["down_bs"][e], inp["down_gs"][e], H, F)
            g, u = Wg @ x[t], Wu @ x[t]
            want[t] += r["w"][t, j] * (Wd @ (g * expit(g) * u))
    assert np.abs(r["out"] - want).max() <= 1e-10 * np.abs(want).max()
    assert np.abs(r["out"] - x).std() > 0.2


def _nearest_ok(target: float, chosen: float, candidates, chosen_code: int, codes) -> bool:
    """chosen is a nearest candidate to target; on a tie, its code is even."""
    dist = np.abs(np.asarray(candidates) - target)
    best = dist.min()
    if abs(chosen - target) != best:
        return False
    tied = [c for c, dd in zip(codes, dist) if dd == best]
    return len(tied) == 1 or chosen_code % 2 == 0


def _check_quantized(x_bits, codes, bs, g):
    rows, cols = x_bits.shape
    x = _bf16(x_bits).astype(np.float32)
    amax = np.float32(np.abs(x).max())
    assert np.float32(g) == amax / np.float32(2688.0)
    e4_codes = list(range(0x7F))
    e4_vals = _e4m3(np.arange(0x7F))
    for r in range(rows):
        for b in range(cols // 16):
            blk = x[r, 16 * b:16 * b + 16]
            bmax = np.float32(np.abs(blk).max())
            t = bmax / (np.float32(6.0) * np.float32(g))
            s = int(bs[r, b])
            if t >= 448:
                assert s == 0x7E
            else:
                assert _nearest_ok(float(t), float(e4_vals[s]), e4_vals, s, e4_codes), (r, b, t, s)
            d = np.float32(e4_vals[s]) * np.float32(g)
            for i in range(16):
                c = int(codes[r, (16 * b + i) // 2] >> (4 * (i % 2))) & 15
                if d == 0:
                    assert c == 0
                    continue
                v = blk[i] / d
                assert (c >> 3) == int(np.signbit(v))
                mag = min(abs(float(v)), 6.0)
                assert _nearest_ok(mag, E2M1[c & 7], E2M1, c & 7, list(range(8))), (r, b, i, v, c)


def test_quantize_decisions_are_nearest():
    x = synth.bf16_matrix(5, 24, 64)
    codes, bs, g = oracle.nvfp4_quantize(x)
    _check_quantized(x, codes, bs, g)


def test_quantize_exact_values_round_trip():
    # blocks whose largest magnitude is the matrix amax (block scale 448) and
    # whose values are E2M1 magnitudes times amax / 6 come back exactly
    rng = np.random.Generator(np.random.PCG64(8))
    vals = np.array(E2M1 + [-v for v in E2M1[1:]], dtype=np.float32)
    x = rng.choice(vals, size=(8, 32)).astype(np.float32)
    x[:, ::16] = 6.0                               # every block reaches the amax
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    codes, bs, g = oracle.nvfp4_quantize(bits)
    assert np.all(bs == 0x7E)
    back = oracle.nvfp4_dequant_matrix(codes, bs, g, 8, 32)
    assert np.abs(back - x).max() <= 1e-6
    _check_quantized(bits, codes, bs, g)


def test_quantize_round_trip_within_half_step():
    x = synth.bf16_matrix(6, 16, 128)
    codes, bs, g = oracle.nvfp4_quantize(x)
    back = oracle.nvfp4_dequant_matrix(codes, bs, g, 16, 128)
    xv = _bf16(x)
    d = np.repeat(_e4m3(bs), 16, axis=1) * g
    # half the widest E2M1 step (4 -> 6) is 1; saturation past 6 adds at most the
    # E4M3 rounding of the block scale (6 * 2^-4 relative)
    assert np.all(np.abs(back - xv) <= 1.0 * d + 1e-12)


def test_quantize_all_zero():
    codes, bs, g = oracle.nvfp4_quantize(np.zeros((2, 32), dtype=np.uint16))
    assert g == 0.0 and not codes.any() and not bs.any()
