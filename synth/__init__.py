"""Seeded synthetic inputs for the qwen3moe MoE FFN (no method arithmetic here).

This module only draws random numbers and lays them out in the byte formats the
method consumes; it computes nothing the method computes.  Both the CPU oracle
(``oracle/``) and the CUDA path take their inputs from here, so that parity is
checked on identical bytes.

Shapes and value distributions follow the Qwen3-30B-A3B file facts given in the
aprender issue "qwen3moe ... has NO working CUDA path" (section "File facts"):
hidden 2048, 128 experts, top-8, expert FFN width 768, router ``ffn_gate_inp``
F32 [128 x 2048], gate/up experts Q4_K, down experts Q6_K or Q4_K, 32 q heads /
4 kv heads, head_dim 128, rope base 1e7, 48 layers.

Recipe (every array is drawn with numpy ``Generator(PCG64(seed))``):

* router weights ~ N(0, 0.02) as float32 [E][H]
* optional per-expert router bias ~ N(0, 1.5) as float32 [E] (prefill workload)
* every k-quant tensor: uniform random bytes for the whole superblock, then the
  fp16 super-scales are overwritten with fp16(|N(0,1)| * 1e-3) (the spread is
  a parameter, 1e-3 unless a case says otherwise)
  (Q4_K: d and dmin; Q6_K: d).  Q6_K's int8 sub-block scales stay uniform bytes.
* activations ~ N(0, 1) as float32.
* decode-step extras: norm weights 1 + 0.1 N(0,1); KV cache entries fp16(N(0,1)).
* NVFP4 experts (E2M1 codes two per byte, an E4M3 scale per 16 elements, an
  fp32 global scale per expert matrix): uniform random code bytes, block scales
  with exponent field uniform in 5..8 and a uniform mantissa, globals
  base * U(0.5, 1.5); BF16 matrices for the quantiser ~ N(0, 0.02) truncated.
* FP8 block-scaled experts (E4M3 codes, one fp32 scale per 128 x 128 block):
  codes with a random sign, a uniform 3-bit mantissa and an exponent field
  rint(N(10, 2.5)) clipped to 0..15 (never the NaN pattern); block scales
  base * U(0.5, 1.5), base 3e-4 for gate/up and 1e-3 for down.

Expert tensors are drawn expert by expert from a stream keyed by
(seed, tensor tag, expert), so that one expert's bytes can be regenerated alone
(the oracle of a 48-layer step regenerates only the experts it routes to).
"""
from __future__ import annotations

import numpy as np

QK_K = 256
BLOCK_BYTES = {"Q4_K": 144, "Q6_K": 210}
QTYPE_CODE = {"Q4_K": 1, "Q6_K": 2}

# tensor tags used to key the per-expert streams
_TAG = {"gate": 1, "up": 2, "down": 3, "wq": 11, "wk": 12, "wv": 13, "wo": 14}


def row_bytes(qtype: str, cols: int) -> int:
    """Bytes of one stored row: cols/256 consecutive superblocks."""
    assert cols % QK_K == 0
    return (cols // QK_K) * BLOCK_BYTES[qtype]


def matrix_bytes(qtype: str, rows: int, cols: int) -> int:
    return rows * row_bytes(qtype, cols)


def _fill_kquant(rng: np.random.Generator, qtype: str, nblocks: int, d_std: float = 1e-3,
                 centered: bool = False) -> np.ndarray:
    """Random superblocks: random bytes, then the fp16 super-scales d (and dmin)
    drawn as |N(0, d_std)|.  centered (Q4_K only): dmin = 7.5 d instead, so that
    the offset dmin * m cancels d * sc * q on average over the uniformly random
    6-bit sc, m and 4-bit q: zero-mean weights, as in a trained model (Q6_K
    weights d * sc * (q - 32) with a signed sc are zero-mean already)."""
    bb = BLOCK_BYTES[qtype]
    raw = np.frombuffer(rng.bytes(nblocks * bb), dtype=np.uint8).reshape(nblocks, bb).copy()
    d = (np.abs(rng.standard_normal(nblocks)) * d_std).astype(np.float16)
    if qtype == "Q4_K":
        dmin = (np.abs(rng.standard_normal(nblocks)) * d_std).astype(np.float16)
        if centered:
            dmin = (d.astype(np.float32) * 7.5).astype(np.float16)
        raw[:, 0:2] = d.view(np.uint8).reshape(nblocks, 2)
        raw[:, 2:4] = dmin.view(np.uint8).reshape(nblocks, 2)
    else:
        raw[:, 208:210] = d.view(np.uint8).reshape(nblocks, 2)
    return raw


def kquant_matrix(seed: int, tag: int, index: int, qtype: str, rows: int, cols: int,
                  d_std: float = 1e-3, centered: bool = False) -> np.ndarray:
    """One quantised matrix [rows][cols] as uint8 [rows][row_bytes]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index])))
    nblk = rows * (cols // QK_K)
    return _fill_kquant(rng, qtype, nblk, d_std, centered).reshape(rows, row_bytes(qtype, cols))


def expert_slice(seed: int, which: str, e: int, qtype: str, rows: int, cols: int,
                 d_std: float = 1e-3, centered: bool = False) -> np.ndarray:
    return kquant_matrix(seed, _TAG[which], e, qtype, rows, cols, d_std, centered)


def expert_tensor(seed: int, which: str, n_experts: int, qtype: str, rows: int, cols: int,
                  d_std: float = 1e-3, centered: bool = False) -> np.ndarray:
    """3-D expert tensor: expert e's slice starts at e * rows * row_bytes (contiguous)."""
    out = np.empty((n_experts, rows, row_bytes(qtype, cols)), dtype=np.uint8)
    for e in range(n_experts):
        out[e] = expert_slice(seed, which, e, qtype, rows, cols, d_std, centered)
    return out


# --------------------------------------------------------------------------- MoE FFN workloads

MOE_CONFIGS = {
    "tiny": dict(name="tiny", H=256, E=8, K=2, F=256, T=4, gate_t="Q4_K", up_t="Q4_K", down_t="Q6_K",
            seed=0, bias_std=None),
    "decode": dict(name="qwen3moe-30b-a3b layer decode T=1", H=2048, E=128, K=8, F=768, T=1,
            gate_t="Q4_K", up_t="Q4_K", down_t="Q6_K", seed=1, bias_std=None),
    "batch8": dict(name="qwen3moe-30b-a3b layer decode T=8, Q4_K down", H=2048, E=128, K=8, F=768, T=8,
            gate_t="Q4_K", up_t="Q4_K", down_t="Q4_K", seed=2, bias_std=None),
    "prefill": dict(name="qwen3moe-30b-a3b layer prefill T=512, biased router", H=2048, E=128, K=8, F=768,
            T=512, gate_t="Q4_K", up_t="Q4_K", down_t="Q6_K", seed=3, bias_std=1.5),
}


def moe_inputs(cfg: dict, T: int | None = None) -> dict:
    """All inputs of one MoE-FFN layer call, drawn in a fixed order.

    Order: router, bias (if any), input activations from the main stream; expert
    tensors from their own per-expert streams.  ``cfg["d_std"]`` (default 1e-3)
    is the spread of the fp16 super-scales; a smaller one gives small expert
    outputs, for cases where the residual must not be negligible.
    """
    H, E, F = cfg["H"], cfg["E"], cfg["F"]
    T = cfg["T"] if T is None else T
    seed = cfg["seed"]
    rng = np.random.Generator(np.random.PCG64(seed))
    router = rng.normal(0.0, 0.02, size=(E, H)).astype(np.float32)
    bias = None
    if cfg.get("bias_std"):
        bias = rng.normal(0.0, cfg["bias_std"], size=E).astype(np.float32)
    x = rng.normal(0.0, 1.0, size=(T, H)).astype(np.float32)
    ds = cfg.get("d_std", 1e-3)
    gate = expert_tensor(seed, "gate", E, cfg["gate_t"], F, H, ds)
    up = expert_tensor(seed, "up", E, cfg["up_t"], F, H, ds)
    down = expert_tensor(seed, "down", E, cfg["down_t"], H, F, ds)
    return dict(H=H, E=E, K=cfg["K"], F=F, T=T, router=router, bias=bias, x=x,
                gate=gate, up=up, down=down,
                gate_t=cfg["gate_t"], up_t=cfg["up_t"], down_t=cfg["down_t"])


# --------------------------------------------------------------------------- FP8 block-scaled experts

FP8_BLOCK = 128
_TAG_FP8 = {"gate": 21, "up": 22, "down": 23}


def _fp8_codes(rng: np.random.Generator, n: int) -> np.ndarray:
    """n random E4M3 codes: random sign, mantissa uniform in 0..7, exponent field
    rint(N(10, 2.5)) clipped to 0..15 (magnitudes spread log-normally around 8,
    up to 448); the NaN pattern S.1111.111 is replaced by S.1111.110."""
    sign = rng.integers(0, 2, size=n, dtype=np.uint8)
    expo = np.clip(np.rint(rng.normal(10.0, 2.5, size=n)), 0, 15).astype(np.uint8)
    mant = rng.integers(0, 8, size=n, dtype=np.uint8)
    mant[(expo == 15) & (mant == 7)] = 6
    return (sign << 7) | (expo << 3) | mant


def fp8_scale_shape(rows: int, cols: int) -> tuple:
    return (-(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK))


def fp8_matrix(seed: int, tag: int, index: int, rows: int, cols: int,
               scale_base: float = 1e-3) -> tuple:
    """One block-scaled FP8 matrix: codes uint8 [rows][cols] and fp32 scales
    [ceil(rows/128)][ceil(cols/128)] = scale_base * U(0.5, 1.5)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index])))
    codes = _fp8_codes(rng, rows * cols).reshape(rows, cols)
    scales = (scale_base * rng.uniform(0.5, 1.5, size=fp8_scale_shape(rows, cols))).astype(np.float32)
    return codes, scales


def fp8_expert_tensor(seed: int, which: str, n_experts: int, rows: int, cols: int,
                      scale_base: float = 1e-3) -> tuple:
    """3-D FP8 expert tensor: codes [E][rows][cols], scales [E][rows/128][cols/128]."""
    rb, cb = fp8_scale_shape(rows, cols)
    codes = np.empty((n_experts, rows, cols), dtype=np.uint8)
    scales = np.empty((n_experts, rb, cb), dtype=np.float32)
    for e in range(n_experts):
        codes[e], scales[e] = fp8_matrix(seed, _TAG_FP8[which], e, rows, cols, scale_base)
    return codes, scales


FP8_CONFIGS = {
    "tiny_fp8": dict(name="tiny, FP8 experts", H=512, E=8, K=2, F=256, T=5, seed=10,
                     gu_scale=6e-4, down_scale=3e-3),
    "decode_fp8": dict(name="qwen3moe-30b-a3b layer decode T=1, FP8 block-scaled experts", H=2048,
                       E=128, K=8, F=768, T=1, seed=11),
}


def moe_inputs_fp8(cfg: dict, T: int | None = None) -> dict:
    """One MoE-FFN layer call over FP8 block-scaled experts: router ~ N(0, 0.02)
    F32 [E][H] and x ~ N(0, 1) from the main stream (as ``moe_inputs``), the
    expert tensors from their own per-expert streams.  Scale bases: gate/up
    ``cfg["gu_scale"]`` (3e-4), down ``cfg["down_scale"]`` (1e-3): gate and up outputs
    of order 1, MoE output of the order of x."""
    H, E, F = cfg["H"], cfg["E"], cfg["F"]
    T = cfg["T"] if T is None else T
    seed = cfg["seed"]
    rng = np.random.Generator(np.random.PCG64(seed))
    router = rng.normal(0.0, 0.02, size=(E, H)).astype(np.float32)
    x = rng.normal(0.0, 1.0, size=(T, H)).astype(np.float32)
    gsb, dsb = cfg.get("gu_scale", 3e-4), cfg.get("down_scale", 1e-3)
    gate, gate_scale = fp8_expert_tensor(seed, "gate", E, F, H, gsb)
    up, up_scale = fp8_expert_tensor(seed, "up", E, F, H, gsb)
    down, down_scale = fp8_expert_tensor(seed, "down", E, H, F, dsb)
    return dict(H=H, E=E, K=cfg["K"], F=F, T=T, router=router, bias=None, x=x, gate=gate,
                gate_scale=gate_scale, up=up, up_scale=up_scale, down=down, down_scale=down_scale)


# --------------------------------------------------------------------------- NVFP4 experts

_TAG_NV = {"gate": 31, "up": 32, "down": 33}


def nvfp4_matrix(seed: int, tag: int, index: int, rows: int, cols: int,
                 global_base: float = 5e-3) -> tuple:
    """One NVFP4 matrix: codes uint8 [rows][cols/2] (uniform random nibbles, every
    E2M1 code equally likely), E4M3 block scales uint8 [rows][cols/16] (positive,
    exponent field uniform in 5..8, mantissa uniform: 0.25 .. 3.75) and a float32
    global scale global_base * U(0.5, 1.5)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index])))
    codes = np.frombuffer(rng.bytes(rows * cols // 2), dtype=np.uint8).reshape(rows, cols // 2).copy()
    expo = rng.integers(5, 9, size=(rows, cols // 16), dtype=np.uint8)
    mant = rng.integers(0, 8, size=(rows, cols // 16), dtype=np.uint8)
    bscale = (expo << 3) | mant
    g = np.float32(global_base * rng.uniform(0.5, 1.5))
    return codes, bscale, g


def nvfp4_expert_tensor(seed: int, which: str, n_experts: int, rows: int, cols: int,
                        global_base: float = 5e-3) -> tuple:
    """3-D NVFP4 expert tensor: codes [E][rows][cols/2], block scales
    [E][rows][cols/16], global scales [E]."""
    codes = np.empty((n_experts, rows, cols // 2), dtype=np.uint8)
    bs = np.empty((n_experts, rows, cols // 16), dtype=np.uint8)
    gs = np.empty(n_experts, dtype=np.float32)
    for e in range(n_experts):
        codes[e], bs[e], gs[e] = nvfp4_matrix(seed, _TAG_NV[which], e, rows, cols, global_base)
    return codes, bs, gs


NVFP4_CONFIGS = {
    "tiny_nvfp4": dict(name="tiny, NVFP4 experts", H=512, E=8, K=2, F=256, T=5, seed=20,
                       gu_global=1e-2, down_global=2e-2),
    "decode_nvfp4": dict(name="qwen3moe-30b-a3b layer decode T=1, NVFP4 experts", H=2048, E=128,
                         K=8, F=768, T=1, seed=21),
}


def moe_inputs_nvfp4(cfg: dict, T: int | None = None) -> dict:
    """One MoE-FFN layer call over NVFP4 experts: router and x as ``moe_inputs``,
    expert tensors from their own per-expert streams.  Global-scale bases:
    gate/up ``cfg["gu_global"]`` (5e-3), down ``cfg["down_global"]`` (1e-2)."""
    H, E, F = cfg["H"], cfg["E"], cfg["F"]
    T = cfg["T"] if T is None else T
    seed = cfg["seed"]
    rng = np.random.Generator(np.random.PCG64(seed))
    router = rng.normal(0.0, 0.02, size=(E, H)).astype(np.float32)
    x = rng.normal(0.0, 1.0, size=(T, H)).astype(np.float32)
    gb, db = cfg.get("gu_global", 5e-3), cfg.get("down_global", 1e-2)
    d = dict(H=H, E=E, K=cfg["K"], F=F, T=T, router=router, bias=None, x=x)
    for which, rows, cols, base in (("gate", F, H, gb), ("up", F, H, gb), ("down", H, F, db)):
        d[which], d[which + "_bs"], d[which + "_gs"] = nvfp4_expert_tensor(seed, which, E, rows,
                                                                            cols, base)
    return d


def bf16_matrix(seed: int, rows: int, cols: int, std: float = 0.02) -> np.ndarray:
    """A BF16 weight matrix ~ N(0, std) as uint16 bit patterns (float32 values
    truncated to their upper 16 bits), the input of the NVFP4 runtime quantiser."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 77])))
    v = rng.normal(0.0, std, size=(rows, cols)).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------- 48-layer decode step

STEP_DEFAULT = dict(n_layers=48, H=2048, E=128, K=8, F=768, n_heads=32, n_kv=4, head_dim=128,
                    ctx=4096, rope_base=1.0e7, eps=1e-6, seed0=100, input_seed=5000)

# one decoder layer of the Qwen3-30B-A3B shape for a batched prefill of 512
# prompt tokens at positions 0..511 (context 4096), with the weight spreads
# under which attention output, MoE output and residual are of one order
PREFILL_LAYER_DEFAULT = dict(STEP_DEFAULT, n_layers=1, T=512, pos0=0, expert_d_std=3e-4,
                             attn_d_std=3e-4, q6_d_scale=0.1, q4_centered=True)


def step_down_qtype(layer: int) -> str:
    """Down-projection quant type of layer i: Q6_K on even layers, Q4_K on odd ones."""
    return "Q6_K" if layer % 2 == 0 else "Q4_K"


def step_layer_small(geo: dict, layer: int) -> dict:
    """Everything of layer i except its expert tensors (norms, attention, router, KV)."""
    H, E = geo["H"], geo["E"]
    hd, nq, nkv, ctx = geo["head_dim"], geo["n_heads"], geo["n_kv"], geo["ctx"]
    seed = geo["seed0"] + layer
    rng = np.random.Generator(np.random.PCG64(seed))
    attn_norm = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    q_norm = (1.0 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    k_norm = (1.0 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    ffn_norm = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    router = rng.normal(0.0, 0.02, size=(E, H)).astype(np.float32)
    k_cache = rng.standard_normal((nkv, ctx, hd)).astype(np.float16)
    v_cache = rng.standard_normal((nkv, ctx, hd)).astype(np.float16)
    ads, cen = geo.get("attn_d_std", 1e-3), geo.get("q4_centered", False)
    wq = kquant_matrix(seed, _TAG["wq"], 0, "Q4_K", nq * hd, H, ads, cen)
    wk = kquant_matrix(seed, _TAG["wk"], 0, "Q4_K", nkv * hd, H, ads, cen)
    wv = kquant_matrix(seed, _TAG["wv"], 0, "Q4_K", nkv * hd, H, ads, cen)
    wo = kquant_matrix(seed, _TAG["wo"], 0, "Q4_K", H, nq * hd, ads, cen)
    return dict(attn_norm=attn_norm, q_norm=q_norm, k_norm=k_norm, ffn_norm=ffn_norm,
                router=router, k_cache=k_cache, v_cache=v_cache, wq=wq, wk=wk, wv=wv, wo=wo,
                down_t=step_down_qtype(layer))


def _expert_d_std(geo: dict, qtype: str) -> float:
    """Spread of the expert super-scales: geo["expert_d_std"] (default 1e-3),
    times geo["q6_d_scale"] (default 1) for Q6_K.  A Q6_K weight is d * sc * q
    with an 8-bit sc and a 6-bit q, about ten times a Q4_K weight at the same d;
    q6_d_scale = 0.1 gives both types the same weight spread."""
    ds = geo.get("expert_d_std", 1e-3)
    return ds * geo.get("q6_d_scale", 1.0) if qtype == "Q6_K" else ds


def step_layer_experts(geo: dict, layer: int) -> dict:
    H, E, F = geo["H"], geo["E"], geo["F"]
    seed = geo["seed0"] + layer
    dt = step_down_qtype(layer)
    cen = geo.get("q4_centered", False)
    return dict(gate=expert_tensor(seed, "gate", E, "Q4_K", F, H, _expert_d_std(geo, "Q4_K"), cen),
                up=expert_tensor(seed, "up", E, "Q4_K", F, H, _expert_d_std(geo, "Q4_K"), cen),
                down=expert_tensor(seed, "down", E, dt, H, F, _expert_d_std(geo, dt), cen))


def step_layer_expert(geo: dict, layer: int, which: str, e: int) -> np.ndarray:
    """Regenerate one expert slice of one layer (identical to the full tensor's slice)."""
    H, F = geo["H"], geo["F"]
    seed = geo["seed0"] + layer
    cen = geo.get("q4_centered", False)
    if which == "down":
        dt = step_down_qtype(layer)
        return expert_slice(seed, "down", e, dt, H, F, _expert_d_std(geo, dt), cen)
    return expert_slice(seed, which, e, "Q4_K", F, H, _expert_d_std(geo, "Q4_K"), cen)


def step_input(geo: dict) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(geo["input_seed"]))
    return rng.standard_normal(geo["H"]).astype(np.float32)


def prefill_input(geo: dict, T: int) -> np.ndarray:
    """Hidden states of T prompt tokens, F32 [T][H], standard normal."""
    rng = np.random.Generator(np.random.PCG64(geo["input_seed"] + 1))
    return rng.standard_normal((T, geo["H"])).astype(np.float32)
