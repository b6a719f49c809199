"""Pin of the oracle's prefill layer (the batched prefill of a whole decoder
layer that the aprender issue "qwen3moe ... has NO working CUDA path" names in
its later gap list, "Prefill is token-by-token"): the token-by-token composition equals a batched formulation written
here from the definition -- all tokens' Q/K/V first, fp16 cache slots, causal
masked softmax attention over the cache and the earlier tokens, O projection,
FFN RMSNorm, routing and the MoE -- using the numpy dequantiser and library
softmax; the norm, RoPE, router and MoE pieces are the separately pinned ones.
"""
import numpy as np
import pytest
import scipy.special

import synth
from oracle import dequant_np
from tests.compare import rel_err

GEO = dict(n_layers=2, H=256, E=8, K=2, F=256, n_heads=4, n_kv=2, head_dim=64, ctx=24,
           rope_base=1.0e7, eps=1e-6, seed0=100, input_seed=5000)


def _batched(o, geo, small, experts, hs, pos0):
    H, hd, nq, nkv = geo["H"], geo["head_dim"], geo["n_heads"], geo["n_kv"]
    T = hs.shape[0]
    eps, base = geo["eps"], geo["rope_base"]
    Wq = dequant_np.dequant("Q4_K", small["wq"], nq * hd, H)
    Wk = dequant_np.dequant("Q4_K", small["wk"], nkv * hd, H)
    Wv = dequant_np.dequant("Q4_K", small["wv"], nkv * hd, H)
    Wo = dequant_np.dequant("Q4_K", small["wo"], H, nq * hd)
    kc = small["k_cache"].astype(np.float16).copy()
    vc = small["v_cache"].astype(np.float16).copy()
    qs = np.zeros((T, nq, hd))
    for i in range(T):
        x = o.rmsnorm(hs[i], small["attn_norm"], eps)
        q, k, v = Wq @ x, Wk @ x, Wv @ x
        for hh in range(nq):
            qs[i, hh] = o.rope_neox(o.rmsnorm(q[hh * hd:(hh + 1) * hd], small["q_norm"], eps),
                                    pos0 + i, base)
        for hh in range(nkv):
            kr = o.rope_neox(o.rmsnorm(k[hh * hd:(hh + 1) * hd], small["k_norm"], eps), pos0 + i, base)
            kc[hh, pos0 + i] = kr.astype(np.float16)
            vc[hh, pos0 + i] = v[hh * hd:(hh + 1) * hd].astype(np.float16)
    grp = nq // nkv
    out = np.zeros((T, H))
    for i in range(T):
        att = np.zeros(nq * hd)
        n = pos0 + i + 1                       # causal: cache and tokens 0..i
        for hh in range(nq):
            K = kc[hh // grp, :n].astype(np.float64)
            V = vc[hh // grp, :n].astype(np.float64)
            p = scipy.special.softmax(K @ qs[i, hh] / np.sqrt(hd))
            att[hh * hd:(hh + 1) * hd] = p @ V
        h = hs[i] + Wo @ att
        x2 = o.rmsnorm(h, small["ffn_norm"], eps)
        _, ids, w, _ = o.route(x2[None, :], small["router"], geo["K"])
        out[i] = o.moe_ffn(x2[None, :], ids, w, experts["gate"], experts["up"], experts["down"],
                           "Q4_K", "Q4_K", small["down_t"], geo["F"], geo["E"], res=h[None, :])[0]
    return out, kc, vc


@pytest.mark.parametrize("layer,pos0,T", [(0, 0, 6), (1, 17, 7)])
def test_token_by_token_equals_batched_causal_layer(oracle_lib, layer, pos0, T):
    small = synth.step_layer_small(GEO, layer)
    experts = synth.step_layer_experts(GEO, layer)
    rng = np.random.default_rng(40 + layer)
    hs = rng.standard_normal((T, GEO["H"]))
    r = oracle_lib.prefill_layer(GEO, small, experts, hs, pos0)
    want, kc, vc = _batched(oracle_lib, GEO, small, experts, hs, pos0)
    assert rel_err(r["h"], want) <= 1e-11
    np.testing.assert_array_equal(r["k_cache"], kc)
    np.testing.assert_array_equal(r["v_cache"], vc)
    # slots outside pos0 .. pos0+T-1 are untouched
    keep = np.ones(GEO["ctx"], bool)
    keep[pos0:pos0 + T] = False
    assert np.array_equal(r["k_cache"][:, keep], small["k_cache"][:, keep])


def test_later_tokens_see_earlier_ones(oracle_lib):
    """Changing the first token changes every later token's output (causal
    attention reaches back), and changing the last changes no earlier one."""
    small = synth.step_layer_small(GEO, 0)
    experts = synth.step_layer_experts(GEO, 0)
    rng = np.random.default_rng(7)
    hs = rng.standard_normal((4, GEO["H"]))
    base = oracle_lib.prefill_layer(GEO, small, experts, hs, 5)["h"]
    h2 = hs.copy()
    h2[0] += 1.0
    a = oracle_lib.prefill_layer(GEO, small, experts, h2, 5)["h"]
    assert all(np.abs(a[i] - base[i]).max() > 1e-9 for i in range(4))
    h3 = hs.copy()
    h3[3] += 1.0
    b = oracle_lib.prefill_layer(GEO, small, experts, h3, 5)["h"]
    assert all(np.array_equal(b[i], base[i]) for i in range(3))


def test_rejects_positions_past_the_context(oracle_lib):
    small = synth.step_layer_small(GEO, 0)
    experts = synth.step_layer_experts(GEO, 0)
    with pytest.raises(ValueError):
        oracle_lib.prefill_layer(GEO, small, experts, np.zeros((3, GEO["H"])), GEO["ctx"] - 2)
