"""Pins of the decoder-layer oracle (48-layer decode step pieces).

Sources: aprender issue "Qwen3 GPU inference produces garbage output"
("Fix Applied": head_dim independent of hidden/heads, GQA uses head_dim,
per-head Q/K RMSNorm); aprender PR "apply per-head Q/K RMSNorm in
forward_qwen3_moe" ("The fix": after bias, before RoPE); SharpInference issue
"Forward-pass divergence on Qwen3-Coder 30B-A3B" (NEOX RoPE pairs offset by
head_dim/2).
"""
import numpy as np
import pytest
import scipy.special

import synth
from tests.compare import rel_err

SMALL = dict(n_layers=2, H=256, E=8, K=2, F=256, n_heads=4, n_kv=2, head_dim=64, ctx=16,
             rope_base=1.0e7, eps=1e-6, seed0=100, input_seed=5000)


def test_rmsnorm_of_constant_vector_is_weight(oracle_lib):
    w = np.random.default_rng(0).standard_normal(128).astype(np.float32)
    for c in (0.5, 3.0, -2.0):
        out = oracle_lib.rmsnorm(np.full(128, c), w, 1e-6)
        exp = np.sign(c) * w.astype(np.float64) / np.sqrt(1 + 1e-6 / c ** 2)
        assert np.allclose(out, exp, rtol=1e-14, atol=0)


def test_rope_position_zero_is_identity(oracle_lib):
    v = np.random.default_rng(1).standard_normal(128)
    assert np.array_equal(oracle_lib.rope_neox(v, 0, 1e7), v)


def test_rope_is_neox_complex_rotation(oracle_lib):
    """NEOX pairing: z_i = v_i + i v_{i+64} rotates by exp(i pos base^(-2i/128))."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal(128)
    for pos in (1, 17, 4095):
        out = oracle_lib.rope_neox(v, pos, 1e7)
        i = np.arange(64)
        z = (v[:64] + 1j * v[64:]) * np.exp(1j * pos * 1e7 ** (-2.0 * i / 128))
        assert np.allclose(out[:64], z.real, rtol=0, atol=1e-12)
        assert np.allclose(out[64:], z.imag, rtol=0, atol=1e-12)
        # pair norms preserved
        assert np.allclose(out[:64] ** 2 + out[64:] ** 2, v[:64] ** 2 + v[64:] ** 2, rtol=1e-13)


def test_attention_single_key_returns_value(oracle_lib):
    rng = np.random.default_rng(3)
    kc = rng.standard_normal((4, 64)).astype(np.float16)
    vc = rng.standard_normal((4, 64)).astype(np.float16)
    out = oracle_lib.attend(rng.standard_normal(64), kc, vc, 0)
    assert np.array_equal(out, vc[0].astype(np.float64))


def test_attention_equal_keys_average_values(oracle_lib):
    rng = np.random.default_rng(4)
    kc = np.tile(rng.standard_normal(64).astype(np.float16), (9, 1))
    vc = rng.standard_normal((9, 64)).astype(np.float16)
    out = oracle_lib.attend(rng.standard_normal(64), kc, vc, 8)
    assert np.allclose(out, vc.astype(np.float64).mean(axis=0), rtol=0, atol=1e-14)


def test_attention_matches_library_softmax(oracle_lib):
    rng = np.random.default_rng(5)
    kc = rng.standard_normal((33, 128)).astype(np.float16)
    vc = rng.standard_normal((33, 128)).astype(np.float16)
    q = rng.standard_normal(128)
    out = oracle_lib.attend(q, kc, vc, 20)
    p = scipy.special.softmax(kc[:21].astype(np.float64) @ q / np.sqrt(128))
    assert np.allclose(out, p @ vc[:21].astype(np.float64), rtol=0, atol=1e-13)


@pytest.fixture(scope="module")
def layer(oracle_lib):
    small = synth.step_layer_small(SMALL, 0)
    experts = synth.step_layer_experts(SMALL, 0)
    h = synth.step_input(SMALL).astype(np.float64)
    return small, experts, h


def test_gqa_mapping_and_cache_write(oracle_lib, layer):
    small, experts, h = layer
    pos = 11
    r = oracle_lib.decode_layer(SMALL, small, experts, h, pos, debug=True)
    hd, nq, nkv = SMALL["head_dim"], SMALL["n_heads"], SMALL["n_kv"]
    grp = nq // nkv
    q = r["q"].reshape(nq, hd)
    att = r["att"].reshape(nq, hd)
    for hq in range(nq):
        kvh = hq // grp
        exp = oracle_lib.attend(q[hq], r["k_cache"][kvh], r["v_cache"][kvh], pos)
        assert np.allclose(att[hq], exp, rtol=0, atol=1e-14)
    # only slot pos is written
    for name in ("k_cache", "v_cache"):
        before, after = small[name], r[name]
        mask = np.ones(SMALL["ctx"], bool)
        mask[pos] = False
        assert np.array_equal(before[:, mask], after[:, mask])
        assert not np.array_equal(before[:, pos], after[:, pos])


def test_qk_norm_precedes_neox_rope(oracle_lib, layer):
    """Undoing the rotation of q must leave RMSNorm(q_raw) * q_norm: per head,
    rms((unrotated q) / q_norm) = 1/sqrt(1 + eps/ms) ~ 1."""
    small, experts, h = layer
    pos = 13
    r = oracle_lib.decode_layer(SMALL, small, experts, h, pos, debug=True)
    hd = SMALL["head_dim"]
    for hq in range(SMALL["n_heads"]):
        qh = r["q"][hq * hd:(hq + 1) * hd]
        un = oracle_lib.rope_neox(qh, -pos, SMALL["rope_base"])
        rms = np.sqrt(np.mean((un / small["q_norm"].astype(np.float64)) ** 2))
        assert abs(rms - 1.0) < 1e-6
        # an interleaved rotation would not undo it
        inter = qh.copy()
        i = np.arange(hd // 2)
        th = -pos * SMALL["rope_base"] ** (-2.0 * i / hd)
        a, b = qh[0::2], qh[1::2]
        inter[0::2] = a * np.cos(th) - b * np.sin(th)
        inter[1::2] = b * np.cos(th) + a * np.sin(th)
        rms_i = np.sqrt(np.mean((inter / small["q_norm"].astype(np.float64)) ** 2))
        assert abs(rms_i - 1.0) > 1e-3


def test_layer_without_attention_weights_is_moe_of_normed_h(oracle_lib, layer):
    small, experts, h = layer
    s = dict(small)
    for n in ("wq", "wk", "wv", "wo"):
        s[n] = np.zeros_like(small[n])
    r = oracle_lib.decode_layer(SMALL, s, experts, h, 7)
    x2 = oracle_lib.rmsnorm(h, small["ffn_norm"], SMALL["eps"])
    _, ids, w, _ = oracle_lib.route(x2, small["router"], SMALL["K"])
    exp = oracle_lib.moe_ffn(x2, ids, w, experts["gate"], experts["up"], experts["down"], "Q4_K",
                             "Q4_K", small["down_t"], SMALL["F"], SMALL["E"], res=h)
    assert np.array_equal(r["ids"], ids[0])
    assert rel_err(r["h"], exp[0]) < 1e-14


def test_layer_without_experts_adds_projected_attention(oracle_lib, layer):
    small, experts, h = layer
    ex = {n: np.zeros_like(v) for n, v in experts.items()}
    r = oracle_lib.decode_layer(SMALL, small, ex, h, 5, debug=True)
    Wo = oracle_lib.dequant_matrix("Q4_K", small["wo"], SMALL["H"],
                                   SMALL["n_heads"] * SMALL["head_dim"])
    assert rel_err(r["h"], h + Wo @ r["att"]) < 1e-13


def test_head_dim_is_independent_of_hidden_over_heads(oracle_lib):
    # Qwen3: q_dim = 32 * 128 = 4096 != hidden 2048 (the page's head_dim fix)
    geo = synth.STEP_DEFAULT
    assert geo["n_heads"] * geo["head_dim"] == 4096 != geo["H"]
    small = synth.step_layer_small(dict(SMALL, H=256, n_heads=4, head_dim=128), 0)
    assert small["wq"].shape[0] == 4 * 128 and small["wo"].shape[1] == synth.row_bytes("Q4_K", 512)


@pytest.mark.parametrize("pos", [0, 17, 39])
def test_step_test_seeds_have_no_topk_near_tie(oracle_lib, pos):
    """The GPU decode-step test demands the kernel's expert ids exactly; that is
    sound only if no layer of its small workload has its K-th and (K+1)-th
    router logits within the fp32 error of each other.  Here they are at least
    1e-2 * max|logit| apart (about 1e4 times the fp32 rounding of a logit)."""
    from tests.test_gpu_decode_step import SMALL as STEP_SMALL
    geo = STEP_SMALL
    h = synth.step_input(geo).astype(np.float64)
    for l in range(geo["n_layers"]):
        small = synth.step_layer_small(geo, l)
        ex = synth.step_layer_experts(geo, l)
        r = oracle_lib.decode_layer(geo, small, ex, h, pos)
        lg = np.sort(r["logits"].astype(np.float64))[::-1]
        K = geo["K"]
        assert lg[K - 1] - lg[K] > 1e-2 * np.abs(lg).max(), (pos, l)
        h = r["h"]
