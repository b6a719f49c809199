"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a number the pages print, a
closed form, a library routine, brute force on tiny inputs or an invariant.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import synth
from oracle import dequant_np
from tests.compare import rel_err

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


# ----------------------------------------------------------------------------- sizes (pages)

def test_expert_strides_match_page_sizes(oracle_lib):
    geo = GOLD["geometry"]
    H, F = geo["hidden"], geo["expert_ffn"]
    eb = GOLD["expert_bytes"]
    assert oracle_lib.expert_stride("Q4_K", F, H) == eb["gate_q4k"] == eb["up_q4k"]
    assert oracle_lib.expert_stride("Q6_K", H, F) == eb["down_q6k"]
    assert oracle_lib.expert_stride("Q4_K", H, F) == eb["down_q4k"]
    assert synth.matrix_bytes("Q4_K", F, H) == eb["gate_q4k"]
    assert synth.matrix_bytes("Q6_K", H, F) == eb["down_q6k"]


def test_expert_total_matches_page_total(oracle_lib):
    geo, eb = GOLD["geometry"], GOLD["expert_bytes"]
    E = geo["n_experts"]
    per_layer_q6 = E * (eb["gate_q4k"] + eb["up_q4k"] + eb["down_q6k"])
    per_layer_q4 = E * (eb["gate_q4k"] + eb["up_q4k"] + eb["down_q4k"])
    total = geo["down_q6k_layers"] * per_layer_q6 + geo["down_q4k_layers"] * per_layer_q4
    assert total == 17_553_162_240
    assert round(total / 1e9, 2) == GOLD["expert_total_gb"]["experts_gb_rounded"]


def test_kv_and_router_sizes():
    geo = GOLD["geometry"]
    kv = GOLD["kv_cache"]
    per_tok = geo["n_layers"] * geo["n_kv_heads"] * geo["head_dim"] * 2 * 4   # K and V, f32
    assert per_tok == kv["bytes_per_token_f32"]
    assert per_tok * 2048 == kv["mib_at_2048"] * 2 ** 20
    assert geo["router_shape"][0] * 4 == GOLD["router_d2h_bytes"]["bytes"]
    assert geo["n_layers"] * geo["top_k"] * 3 == GOLD["upload_per_token"]["uploads"]
    # about 1 GB/token: 48 layers x 8 experts x average expert slice
    eb = GOLD["expert_bytes"]
    avg = (eb["gate_q4k"] + eb["up_q4k"] + (eb["down_q6k"] + eb["down_q4k"]) / 2)
    assert abs(geo["n_layers"] * geo["top_k"] * avg / 1e9 - 1.0) < 0.15


# ----------------------------------------------------------------------------- fp16 (library)

def test_half_to_double_exhaustive(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.half_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_double_to_half_matches_numpy(oracle_lib):
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
                           [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -24, 2.0 ** -25,
                            3 * 2.0 ** -26, 2.0 ** -14 - 2.0 ** -26, 1.0 + 2.0 ** -11,
                            1.0 + 3 * 2.0 ** -11]])
    for v in vals:
        assert oracle_lib.double_to_half_bits(v) == int(np.float16(v).view(np.uint16)), v


# ----------------------------------------------------------------------------- k-quant blocks

def _pack_q4k_scales(s, m):
    """Independent packer for the 12-byte Q4_K scale field (inverse of the format)."""
    sc = np.zeros(12, dtype=np.uint8)
    for j in range(8):
        if j < 4:
            sc[j] |= s[j] & 63
            sc[j + 4] |= m[j] & 63
        else:
            sc[j + 4] |= (s[j] & 15) | ((m[j] & 15) << 4)
            sc[j - 4] |= (s[j] >> 4) << 6
            sc[j] |= (m[j] >> 4) << 6
    return sc


def _q4k_block(d, dmin, s, m, nib):
    """nib: [8][32] values 0..15 (sub-block, position)."""
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    blk[4:16] = _pack_q4k_scales(s, m)
    for c in range(4):
        blk[16 + 32 * c:16 + 32 * c + 32] = nib[2 * c] | (nib[2 * c + 1] << 4)
    return blk


def test_q4k_unit_scale_block_returns_nibbles(oracle_lib):
    rng = np.random.default_rng(1)
    nib = rng.integers(0, 16, (8, 32)).astype(np.uint8)
    blk = _q4k_block(1.0, 0.0, [1] * 8, [0] * 8, nib)
    y = oracle_lib.dequant_block("Q4_K", blk)
    assert np.array_equal(y, nib.reshape(-1).astype(np.float64))


def test_q4k_constant_block_closed_form(oracle_lib):
    rng = np.random.default_rng(2)
    for _ in range(50):
        s = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        c = int(rng.integers(0, 16))
        d, dmin = float(np.float16(rng.random())), float(np.float16(rng.random()))
        blk = _q4k_block(d, dmin, s, m, np.full((8, 32), c, dtype=np.uint8))
        y = oracle_lib.dequant_block("Q4_K", blk).reshape(8, 32)
        for j in range(8):
            assert np.all(y[j] == d * s[j] * c - dmin * m[j])


def test_q4k_all_scale_min_pairs_roundtrip(oracle_lib):
    # every 6-bit scale and min reaches the right sub-block (one-hot d=1, dmin=1)
    for j in range(8):
        for v in (0, 1, 15, 16, 47, 63):
            s = [0] * 8
            m = [0] * 8
            s[j] = v
            m[(j + 3) % 8] = 63 - v
            blk = _q4k_block(1.0, 1.0, s, m, np.ones((8, 32), dtype=np.uint8))
            y = oracle_lib.dequant_block("Q4_K", blk).reshape(8, 32)
            exp = np.array([s[i] * 1 - m[i] for i in range(8)], dtype=np.float64)
            assert np.array_equal(y[:, 0], exp)


def _q6k_block(d, sc, q6):
    """q6: [256] values 0..63 in element order; sc: 16 int8."""
    q6 = np.asarray(q6).reshape(2, 4, 32)
    blk = np.zeros(210, dtype=np.uint8)
    for n in range(2):
        lo = q6[n] & 15
        hi = q6[n] >> 4
        blk[64 * n:64 * n + 32] = lo[0] | (lo[2] << 4)
        blk[64 * n + 32:64 * n + 64] = lo[1] | (lo[3] << 4)
        blk[128 + 32 * n:128 + 32 * n + 32] = hi[0] | (hi[1] << 2) | (hi[2] << 4) | (hi[3] << 6)
    blk[192:208] = np.asarray(sc, dtype=np.int8).view(np.uint8)
    blk[208:210] = np.array([d], dtype=np.float16).view(np.uint8)
    return blk


def test_q6k_unit_scale_block_returns_q_minus_32(oracle_lib):
    rng = np.random.default_rng(3)
    q6 = rng.integers(0, 64, 256)
    blk = _q6k_block(1.0, [1] * 16, q6)
    y = oracle_lib.dequant_block("Q6_K", blk)
    assert np.array_equal(y, (q6 - 32).astype(np.float64))


def test_q6k_scale_per_16_and_sign(oracle_lib):
    rng = np.random.default_rng(4)
    q6 = np.full(256, 40)
    sc = rng.integers(-128, 128, 16)
    d = float(np.float16(0.5))
    y = oracle_lib.dequant_block("Q6_K", _q6k_block(d, sc, q6))
    # element i = 128n + 32g + l uses scale 8n + l//16 + 2g
    for i in range(256):
        n, g, l = i // 128, (i % 128) // 32, i % 32
        assert y[i] == d * sc[8 * n + l // 16 + 2 * g] * 8


def test_numpy_and_c_dequant_agree_bit_for_bit(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    H, F = inp["H"], inp["F"]
    for e in range(inp["E"]):
        for name, qt, rows, cols in (("gate", "Q4_K", F, H), ("up", "Q4_K", F, H),
                                     ("down", inp["down_t"], H, F)):
            a = oracle_lib.dequant_matrix(qt, inp[name][e], rows, cols)
            b = dequant_np.dequant(qt, inp[name][e], rows, cols)
            assert np.array_equal(a, b), (name, e)


def test_subnormal_scales_occur_and_decode(oracle_lib):
    # d = fp16(|N|*1e-3) is subnormal below 6.1e-5: the generator produces some
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    d = inp["gate"].reshape(-1, 144)[:, 0:2].copy().view(np.float16).reshape(-1)
    assert np.any((d != 0) & (np.abs(d.astype(np.float64)) < 2 ** -14))


# ----------------------------------------------------------------------------- router

def _route(oracle_lib, x, router, K, bias=None, norm=True):
    return oracle_lib.route(x, router, K, bias, norm)


def test_router_logits_are_f32_rounded_matmul(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    logits, ids, w, probs = _route(oracle_lib, inp["x"], inp["router"], 8)
    ref = inp["x"].astype(np.float64) @ inp["router"].astype(np.float64).T
    # exact double dot rounded to f32 may differ from numpy's BLAS order by 1 ulp at most
    assert np.all(np.abs(logits - ref.astype(np.float32)) <= np.spacing(np.abs(ref).astype(np.float32)))


def test_router_weights_sum_to_one_and_order(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    logits, ids, w, probs = _route(oracle_lib, inp["x"], inp["router"], 8)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-12)
    for t in range(ids.shape[0]):
        lg = logits[t]
        sel = lg[ids[t]]
        assert np.all(np.diff(sel) <= 0)
        rest = np.delete(lg, ids[t])
        assert sel.min() >= rest.max()
        # w proportional to exp(logit) over the selected set (library softmax)
        assert np.allclose(w[t], scipy.special.softmax(sel.astype(np.float64)), rtol=0, atol=1e-15)


def test_router_k1_gives_weight_one(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["decode"])
    logits, ids, w, probs = _route(oracle_lib, inp["x"], inp["router"], 1)
    assert w[0, 0] == 1.0
    assert ids[0, 0] == int(np.argmax(logits[0]))


def test_router_k_equals_e_is_dense_softmax(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    E = inp["E"]
    logits, ids, w, probs = _route(oracle_lib, inp["x"], inp["router"], E)
    for t in range(inp["T"]):
        p = scipy.special.softmax(logits[t].astype(np.float64))
        assert np.allclose(w[t], p[ids[t]], rtol=1e-13, atol=0)
        assert sorted(ids[t].tolist()) == list(range(E))


def test_router_equal_logits_pick_lowest_indices(oracle_lib):
    x = np.ones((2, 256), dtype=np.float32)
    router = np.zeros((16, 256), dtype=np.float32)
    logits, ids, w, probs = _route(oracle_lib, x, router, 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 2
    assert np.all(w == 0.25)


def test_router_without_renorm_gives_softmax_probs(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    logits, ids, w, probs = _route(oracle_lib, inp["x"], inp["router"], 8, norm=False)
    for t in range(inp["T"]):
        p = scipy.special.softmax(logits[t].astype(np.float64))
        assert np.allclose(w[t], p[ids[t]], rtol=1e-13, atol=0)


def test_router_bias_shifts_selection(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    bias = np.zeros(inp["E"], dtype=np.float32)
    bias[5] = 100.0
    logits, ids, w, probs = _route(oracle_lib, inp["x"], inp["router"], 2, bias=bias)
    assert np.all(ids[:, 0] == 5)


# ----------------------------------------------------------------------------- FFN

def test_ffn_brute_force_dense_config1(oracle_lib):
    """Dense evaluation of every expert for every token, combined through a
    top-k mask, equals the sparse oracle (config 1)."""
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    H, F, E, K, T = inp["H"], inp["F"], inp["E"], inp["K"], inp["T"]
    r = oracle_lib.moe_forward(inp)
    x = inp["x"].astype(np.float64)
    Y = np.zeros((T, E, H))
    for e in range(E):
        Wg = dequant_np.dequant("Q4_K", inp["gate"][e], F, H)
        Wu = dequant_np.dequant("Q4_K", inp["up"][e], F, H)
        Wd = dequant_np.dequant(inp["down_t"], inp["down"][e], H, F)
        g = x @ Wg.T
        u = x @ Wu.T
        a = g * scipy.special.expit(g) * u
        Y[:, e, :] = a @ Wd.T
    # gate mask from the library softmax of the F32 logits
    mask = np.zeros((T, E))
    for t in range(T):
        p = scipy.special.softmax(r["logits"][t].astype(np.float64))
        top = np.argsort(-r["logits"][t], kind="stable")[:K]
        mask[t, top] = p[top] / p[top].sum()
    dense = x + np.einsum("te,teh->th", mask, Y)
    assert rel_err(r["out"], dense) < 1e-12


def test_ffn_expert_permutation_invariance(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    r = oracle_lib.moe_forward(inp)
    perm = np.random.default_rng(5).permutation(inp["E"])
    inv = np.argsort(perm)
    p = dict(inp)
    for n in ("router", "gate", "up", "down"):
        p[n] = np.ascontiguousarray(inp[n][perm])
    r2 = oracle_lib.moe_forward(p)
    assert np.array_equal(perm[r2["ids"]], r["ids"])
    assert rel_err(r2["out"], r["out"]) < 1e-13


def test_ffn_batch_independence(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    r = oracle_lib.moe_forward(inp)
    for t in (0, 5):
        one = dict(inp)
        one["x"] = inp["x"][t:t + 1]
        one["T"] = 1
        r1 = oracle_lib.moe_forward(one)
        assert np.array_equal(r1["ids"][0], r["ids"][t])
        assert np.array_equal(r1["out"][0], r["out"][t])


def test_ffn_zero_experts_returns_residual(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["tiny"])
    p = dict(inp)
    for n in ("gate", "up", "down"):
        p[n] = np.zeros_like(inp[n])
    r = oracle_lib.moe_forward(p)
    assert np.array_equal(r["out"], inp["x"].astype(np.float64))


def test_ffn_silu_closed_form_single_expert(oracle_lib):
    """One expert whose gate/up rows dequantise to constants: g = u = c * sum(x)."""
    H = F = 256
    d = 1.0 / 64
    blk = _q4k_block(d, 0.0, [1] * 8, [0] * 8, np.full((8, 32), 2, dtype=np.uint8))
    gate = np.tile(blk, (1, F, 1)).reshape(1, F, 144)
    dblk = _q6k_block(1.0 / 256, [1] * 16, np.full(256, 33))       # every weight = 1/256
    down = np.tile(dblk, (1, H, 1)).reshape(1, H, 210)
    x = np.random.default_rng(6).standard_normal((1, H)).astype(np.float32)
    out = oracle_lib.moe_ffn(x, np.zeros((1, 1), np.int32), np.ones((1, 1)), gate, gate, down,
                             "Q4_K", "Q4_K", "Q6_K", F, 1)
    g = 2 * d * x.astype(np.float64).sum()
    a = g / (1 + np.exp(-g)) * g
    exp = x.astype(np.float64) + F * a / 256
    assert rel_err(out, exp) < 1e-13
