"""The comparator must reject the routing and dequant faults the pages inject.

Mirrors the aprender issue "qwen3moe ... has NO working CUDA path", R1 receipt
("The oracle bites"): after a clean control, WrongExpert, DropTopExpert and
UniformWeights must all be rejected.  A nibble-half swap in the dequant is added.
The mutants are planted in the oracle's output, on the CPU.
"""
import numpy as np
import pytest

import synth
from tests.compare import TOL_FP32, TOL_W, ids_match, min_gap, rel_err, tie_bound


@pytest.fixture(scope="module")
def case(oracle_lib):
    inp = synth.moe_inputs(synth.MOE_CONFIGS["batch8"])
    ref = oracle_lib.moe_forward(inp)
    bound = tie_bound(ref["logits"])
    return inp, ref, bound


def _ffn(oracle_lib, inp, ids, w, gate=None):
    return oracle_lib.moe_ffn(inp["x"], ids, w, inp["gate"] if gate is None else gate, inp["up"],
                              inp["down"], inp["gate_t"], inp["up_t"], inp["down_t"], inp["F"],
                              inp["E"])


def test_clean_control_passes(oracle_lib, case):
    inp, ref, bound = case
    out = _ffn(oracle_lib, inp, ref["ids"], ref["w"])
    ok, ties = ids_match(ref["ids"], ref["ids"], ref["logits"], bound)
    assert ok and not ties
    assert rel_err(out, ref["out"]) < 1e-15


def test_wrong_expert_rejected(oracle_lib, case):
    inp, ref, bound = case
    ids = ref["ids"].copy()
    for t in range(ids.shape[0]):
        order = np.argsort(-ref["logits"][t], kind="stable")
        ids[t, 0] = order[inp["K"] + 3]          # an expert well outside the top-k
    ok, _ = ids_match(ids, ref["ids"], ref["logits"], bound)
    assert not ok
    out = _ffn(oracle_lib, inp, ids, ref["w"])
    assert rel_err(out, ref["out"]) > TOL_FP32


def test_drop_top_expert_rejected(oracle_lib, case):
    inp, ref, bound = case
    ids = ref["ids"][:, 1:]
    w = ref["w"][:, 1:] / ref["w"][:, 1:].sum(axis=1, keepdims=True)
    out = _ffn(oracle_lib, inp, ids, w)
    assert rel_err(out, ref["out"]) > TOL_FP32
    padded = np.concatenate([ids, ids[:, :1]], axis=1)
    ok, _ = ids_match(padded, ref["ids"], ref["logits"], bound)
    assert not ok


def test_uniform_weights_rejected(oracle_lib, case):
    inp, ref, bound = case
    w = np.full_like(ref["w"], 1.0 / inp["K"])
    assert np.abs(w - ref["w"]).max() > TOL_W
    out = _ffn(oracle_lib, inp, ref["ids"], w)
    assert rel_err(out, ref["out"]) > TOL_FP32


def test_nibble_half_swap_rejected(oracle_lib, case):
    inp, ref, bound = case
    g = inp["gate"].reshape(-1, 144).copy()
    q = g[:, 16:144]
    g[:, 16:144] = ((q & 15) << 4) | (q >> 4)
    out = _ffn(oracle_lib, inp, ref["ids"], ref["w"], gate=g.reshape(inp["gate"].shape))
    assert rel_err(out, ref["out"]) > TOL_FP32


def test_near_tie_swap_accepted_only_within_bound(oracle_lib):
    logits = np.array([[3.0, 2.0, 1.0, 1.0 + 1e-7, 0.0]])
    ref = np.array([[0, 1, 3]])
    swapped = np.array([[0, 1, 2]])
    assert ids_match(swapped, ref, logits, 1e-6)[0]
    assert not ids_match(swapped, ref, logits, 1e-8)[0]


def test_tie_bound_is_far_below_the_fixed_seed_gaps(oracle_lib):
    """At the fixed seeds of the MoE workloads, the smallest gap between adjacent
    logits among each token's top k+1 exceeds the near-tie allowance, so the
    GPU tests there can require exactly the oracle's ordered ids."""
    for cid in ("tiny", "decode", "batch8", "prefill"):
        inp = synth.moe_inputs(synth.MOE_CONFIGS[cid])
        lg = inp["x"].astype(np.float64) @ inp["router"].astype(np.float64).T
        if inp["bias"] is not None:
            lg = lg + inp["bias"].astype(np.float64)
        srt = np.sort(lg, axis=1)[:, ::-1][:, :inp["K"] + 1]
        gaps = -np.diff(srt, axis=1)
        assert np.all(gaps.min(axis=1) > tie_bound(lg)), cid
        assert min_gap(lg, inp["K"]) > 0
