"""Pins of the oracle's Q8_K-activation variant (the int8-activation expert GEMVs
named in the aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA
path", section "Gaps ... G8" and the R1 receipt's Q8_K measurement).

What fixes each expected value: invariants of the block format (group sums,
code range, the largest value on code -128, the rounding bound), exact
representability (powers of two), the independent numpy dequantiser, and the
composition of separately pinned parts.  No expected value here is the
oracle's formula typed again.
"""
import numpy as np
import pytest

import synth
from oracle import dequant_np
from tests.compare import rel_err


def _blocks(rng, n, scale=1.0):
    return (rng.standard_normal(n) * scale).astype(np.float32)


# ----------------------------------------------------------------------------- quantiser

def test_group_sums_and_code_range(oracle_lib):
    rng = np.random.default_rng(11)
    x = _blocks(rng, 256 * 8, 3.0)
    d, q, bs = oracle_lib.q8k_quantize(x)
    assert d.shape == (8,) and q.shape == (2048,) and bs.shape == (128,)
    np.testing.assert_array_equal(bs.astype(np.int64), q.astype(np.int64).reshape(-1, 16).sum(axis=1))
    assert q.min() >= -128 and q.max() <= 127


def test_largest_value_takes_code_minus_128_and_is_exact(oracle_lib):
    rng = np.random.default_rng(12)
    x = _blocks(rng, 256 * 4)
    x[5] = 7.25            # block 0: positive extreme
    x[256 + 9] = -9.5      # block 1: negative extreme
    d, q, _ = oracle_lib.q8k_quantize(x)
    for b, i in ((0, 5), (1, 256 + 9)):
        assert q[i] == -128
        assert np.float32(d[b]) * np.float32(-128) == x[i]      # d = -v/128, a power-of-two step
    # the sign of d is opposite to the extreme value's
    assert d[0] < 0 < d[1]


def test_rounding_error_bound(oracle_lib):
    """Every value is within half a step of d*q, except those clamped from +128
    to 127 (the opposite extreme of a block), which are within one step."""
    rng = np.random.default_rng(13)
    x = _blocks(rng, 256 * 32, 2.0)
    x[300] = -x[300 - 1]   # a few exact opposites of other values
    d, q, _ = oracle_lib.q8k_quantize(x)
    step = np.abs(np.repeat(d, 256)).astype(np.float64)
    err = np.abs(x.astype(np.float64) - np.repeat(d, 256).astype(np.float64) * q)
    clamped = (q == 127) & (err > 0.5 * step * (1 + 1e-5))
    assert np.all(err[~clamped] <= 0.5 * step[~clamped] * (1 + 1e-5))
    assert np.all(err[clamped] <= step[clamped] * (1 + 1e-5))


def test_exactly_representable_values_round_trip(oracle_lib):
    """x = c*k with c a power of two and integer codes k (k[0] = -128 the extreme):
    the scale is exactly c and every code is k."""
    rng = np.random.default_rng(14)
    k = rng.integers(-127, 128, size=256)
    k[0] = -128
    for c in (2.0 ** -7, 1.0, 2.0 ** 5):
        x = (k * c).astype(np.float32)
        d, q, bs = oracle_lib.q8k_quantize(x)
        assert d[0] == np.float32(c)
        np.testing.assert_array_equal(q.astype(np.int64), k)
        assert bs.sum() == k.sum()


def test_zero_block_and_power_of_two_scaling(oracle_lib):
    rng = np.random.default_rng(15)
    x = _blocks(rng, 512)
    x[:256] = 0.0
    d, q, bs = oracle_lib.q8k_quantize(x)
    assert d[0] == 0.0 and not q[:256].any() and not bs[:16].any()
    # scaling the input by a power of two scales d and keeps the codes
    d2, q2, _ = oracle_lib.q8k_quantize(x * np.float32(8.0))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(d2, d * np.float32(8.0))


def test_rejects_partial_blocks(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.q8k_quantize(np.ones(300, dtype=np.float32))


# ----------------------------------------------------------------------------- integer dot

@pytest.mark.parametrize("qtype", ["Q4_K", "Q6_K"])
def test_integer_dot_equals_dequantised_dot(oracle_lib, qtype):
    """The integer form (sub-block sums, code-group sums for the Q4_K minimum
    term, int8 scales for Q6_K) equals the plain dot of the independently
    dequantised weights with the dequantised activations."""
    cols, rows = 1024, 6
    raw = synth.kquant_matrix(21, 7, 0, qtype, rows, cols)
    W = dequant_np.dequant(qtype, raw, rows, cols)
    rb = synth.row_bytes(qtype, cols)
    rng = np.random.default_rng(16)
    x = _blocks(rng, cols, 1.5)
    q8 = oracle_lib.q8k_quantize(x)
    xq = np.repeat(q8[0], 256).astype(np.float64) * q8[1]
    for r in range(rows):
        got = oracle_lib.q8k_dot(qtype, raw.reshape(-1)[r * rb:(r + 1) * rb], cols, q8)
        want = float(np.dot(W[r], xq))
        assert abs(got - want) <= 1e-12 * max(1.0, np.abs(W[r]).dot(np.abs(xq)))


def test_q4k_min_term_uses_the_code_sums(oracle_lib):
    """A Q4_K row whose codes are all zero reduces to -dmin * sum_j m_j * B_j * dx:
    the dot then depends on the activations only through the 32-value code sums."""
    cols = 256
    raw = synth.kquant_matrix(22, 7, 0, "Q4_K", 1, cols).reshape(-1).copy()
    raw[16:144] = 0                       # every 4-bit code 0
    W = dequant_np.dequant("Q4_K", raw, 1, cols)[0]
    assert np.all(W.reshape(8, 32) == W.reshape(8, 32)[:, :1])   # constant per sub-block
    rng = np.random.default_rng(17)
    x = _blocks(rng, cols)
    q8 = oracle_lib.q8k_quantize(x)
    got = oracle_lib.q8k_dot("Q4_K", raw, cols, q8)
    sub = q8[1].astype(np.int64).reshape(8, 32).sum(axis=1)
    want = float(q8[0][0]) * float(np.dot(W.reshape(8, 32)[:, 0], sub))
    assert abs(got - want) <= 1e-12 * max(1.0, abs(want))


# ----------------------------------------------------------------------------- layer

def test_layer_is_the_composition_of_pinned_parts(oracle_lib):
    """moe_ffn_q8k on the small geometry equals its steps done here with the
    pinned quantiser and the independent numpy dequantiser."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    H, F, E, K = inp["H"], inp["F"], inp["E"], inp["K"]
    _, ids, w, _ = oracle_lib.route(inp["x"], inp["router"], K)
    got = oracle_lib.moe_ffn_q8k(inp["x"], ids, w, inp["gate"], inp["up"], inp["down"],
                                 inp["gate_t"], inp["up_t"], inp["down_t"], F, E)
    sg = synth.matrix_bytes(inp["gate_t"], F, H)
    sd = synth.matrix_bytes(inp["down_t"], H, F)
    want = inp["x"].astype(np.float64).copy()
    for t in range(inp["T"]):
        dx, qx, _ = oracle_lib.q8k_quantize(inp["x"][t])
        xq = np.repeat(dx, 256).astype(np.float64) * qx
        for j in range(K):
            e = int(ids[t, j])
            Wg = dequant_np.dequant(inp["gate_t"], inp["gate"].reshape(-1)[e * sg:(e + 1) * sg], F, H)
            Wu = dequant_np.dequant(inp["up_t"], inp["up"].reshape(-1)[e * sg:(e + 1) * sg], F, H)
            Wd = dequant_np.dequant(inp["down_t"], inp["down"].reshape(-1)[e * sd:(e + 1) * sd], H, F)
            g, u = Wg @ xq, Wu @ xq
            a = g / (1.0 + np.exp(-g)) * u
            da, qa, _ = oracle_lib.q8k_quantize(a.astype(np.float32))
            want[t] += w[t, j] * (Wd @ (np.repeat(da, 256).astype(np.float64) * qa))
    assert rel_err(got, want) <= 1e-10


def test_int8_activations_move_the_layer_output_a_little(oracle_lib):
    """Against the fp64-activation layer the Q8_K variant differs (it quantises)
    but stays close (8-bit codes per 256 values)."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    F, E, K = inp["F"], inp["E"], inp["K"]
    _, ids, w, _ = oracle_lib.route(inp["x"], inp["router"], K)
    args = (inp["x"], ids, w, inp["gate"], inp["up"], inp["down"], inp["gate_t"], inp["up_t"],
            inp["down_t"], F, E)
    exact = oracle_lib.moe_ffn(*args) - inp["x"]
    q8 = oracle_lib.moe_ffn_q8k(*args) - inp["x"]
    err = rel_err(q8, exact)
    assert 1e-4 < err < 5e-2
