"""CPU oracle of the qwen3moe MoE FFN over GGUF k-quant experts (double precision).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg may import this package; the product path never does.  It
shares no code with the CUDA path; both take their inputs from ``synth``.

The arithmetic lives in ``qmoe_oracle.c`` (plain C, every quantity in double,
serial sums in index order).  ``dequant_np`` is a second, independent numpy
dequantiser used only to cross-check the C one.

Sources: aprender issue "qwen3moe (Qwen3-30B-A3B, Qwen3-Coder-30B-A3B, Q4_K_M)
has NO working CUDA path" (sections "File facts", "Gaps ... G3"); aprender issue
"Qwen3 GPU inference produces garbage output" ("Fix Applied"); aprender PR
"apply per-head Q/K RMSNorm in forward_qwen3_moe" ("The fix"); SharpInference
issue "Forward-pass divergence on Qwen3-Coder 30B-A3B" (closing comment).

Parity status: every function here is pinned by a ``-m "not gpu"`` test (closed
forms, library routines, brute force, invariants); the 48-layer composition as a
whole is pinned only through its pinned parts.  The Q8_K-activation functions
(``q8k_quantize``, ``q8k_dot``, ``moe_ffn_q8k``) follow a reading of a format the
pages name without defining (the GGUF 8-bit activation block); they are pinned
by invariants, exact cases and the independent numpy dequantiser.  ``prefill_layer``
is pinned against a batched causal formulation written in the tests.  The FP8
functions (``fp8_e4m3_to_double``, ``fp8_dequant_matrix``, ``moe_ffn_fp8``) are
pinned against the E4M3 definition, torch's float8_e4m3fn conversion and a
dense numpy brute force (atlasinference source page
"spark_model/weight_loader/qwen3.rs", load_layers: FP8 block-128 weights).  The
NVFP4 functions (``e2m1_to_double``, ``nvfp4_dequant_matrix``, ``moe_ffn_nvfp4``,
``nvfp4_quantize``) are pinned against the E2M1 value table, torch's E4M3
conversion, a numpy brute force, and brute-force optimality of every rounding
decision of the quantiser (same page: BF16 -> NVFP4 runtime quantisation).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libqmoe_oracle.so")
_lock = threading.Lock()
_lib = None

Q4_K, Q6_K = 1, 2
QCODE = {"Q4_K": Q4_K, "Q6_K": Q6_K}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _p(a, t):
    return None if a is None else a.ctypes.data_as(C.POINTER(t))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            dp, fp, ip, up8, u16 = (C.POINTER(C.c_double), C.POINTER(C.c_float),
                                    C.POINTER(C.c_int32), C.POINTER(C.c_uint8),
                                    C.POINTER(C.c_uint16))
            L.qo_half_to_double.argtypes = [C.c_uint16]
            L.qo_half_to_double.restype = C.c_double
            L.qo_double_to_half.argtypes = [C.c_double]
            L.qo_double_to_half.restype = C.c_uint16
            L.qo_block_bytes.argtypes = [C.c_int]
            L.qo_expert_stride.argtypes = [C.c_int, C.c_long, C.c_long]
            L.qo_expert_stride.restype = C.c_long
            L.qo_dequant_block.argtypes = [C.c_int, up8, dp]
            L.qo_dequant_matrix.argtypes = [C.c_int, up8, C.c_long, C.c_long, dp]
            L.qo_router.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, dp, fp, fp, ip,
                                    fp, ip, dp, dp]
            L.qo_moe_ffn.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, dp, dp, ip, dp,
                                     up8, C.c_int, up8, C.c_int, up8, C.c_int, dp, dp, dp]
            L.qo_rmsnorm.argtypes = [C.c_long, dp, fp, C.c_double, dp]
            L.qo_rope_neox.argtypes = [C.c_int, dp, C.c_int, C.c_double]
            L.qo_attend.argtypes = [C.c_int, dp, u16, u16, C.c_int, dp]
            i8p, i16p = C.POINTER(C.c_int8), C.POINTER(C.c_int16)
            L.qo_q8k_quantize.argtypes = [C.c_long, fp, fp, i8p, i16p]
            L.qo_dot_q8k.argtypes = [C.c_int, up8, C.c_long, fp, i8p, i16p]
            L.qo_dot_q8k.restype = C.c_double
            L.qo_moe_ffn_q8k.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, dp, dp, ip,
                                         dp, up8, C.c_int, up8, C.c_int, up8, C.c_int, dp, dp]
            L.qo_fp8_e4m3_to_double.argtypes = [C.c_uint8]
            L.qo_fp8_e4m3_to_double.restype = C.c_double
            L.qo_fp8_dequant_matrix.argtypes = [up8, fp, C.c_long, C.c_long, dp]
            L.qo_fp8_scale_count.argtypes = [C.c_long, C.c_long]
            L.qo_fp8_scale_count.restype = C.c_long
            L.qo_moe_ffn_fp8.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, dp, dp, ip,
                                         dp, up8, fp, up8, fp, up8, fp, dp, dp, dp]
            L.qo_e2m1_to_double.argtypes = [C.c_uint8]
            L.qo_e2m1_to_double.restype = C.c_double
            L.qo_nvfp4_dequant_matrix.argtypes = [up8, up8, C.c_float, C.c_long, C.c_long, dp]
            L.qo_moe_ffn_nvfp4.argtypes = ([C.c_int] * 5 + [dp, dp, ip, dp] + [up8, up8, fp] * 3
                                           + [dp, dp, dp])
            L.qo_nvfp4_quantize.argtypes = [C.c_long, C.c_long, u16, up8, up8, fp]
            L.qo_decode_layer.argtypes = (
                [C.c_int] * 8 + [C.c_double, C.c_double, C.c_int, dp] + [fp] * 4 + [up8] * 4
                + [fp, up8, up8, up8, C.c_int, u16, u16, ip, fp, ip, dp, dp, dp])
            _lib = L
    return _lib


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


# ----------------------------------------------------------------------------- fp16 / dequant

def half_to_double(bits: int) -> float:
    return lib().qo_half_to_double(int(bits))


def double_to_half_bits(v: float) -> int:
    return lib().qo_double_to_half(float(v))


def expert_stride(qtype: str, rows: int, cols: int) -> int:
    return lib().qo_expert_stride(QCODE[qtype], rows, cols)


def dequant_block(qtype: str, blk: np.ndarray) -> np.ndarray:
    blk = _u8(blk).reshape(-1)
    out = np.empty(256, dtype=np.float64)
    rc = lib().qo_dequant_block(QCODE[qtype], _p(blk, C.c_uint8), _p(out, C.c_double))
    if rc:
        raise ValueError("bad qtype")
    return out


def dequant_matrix(qtype: str, data: np.ndarray, rows: int, cols: int) -> np.ndarray:
    data = _u8(data).reshape(-1)
    out = np.empty((rows, cols), dtype=np.float64)
    rc = lib().qo_dequant_matrix(QCODE[qtype], _p(data, C.c_uint8), rows, cols, _p(out, C.c_double))
    if rc:
        raise ValueError("dequant_matrix failed")
    return out


# ----------------------------------------------------------------------------- router / FFN

def route(x, router, K, bias=None, norm_topk=True, force=None):
    """Returns (logits f32 [T][E], ids int32 [T][K], w f64 [T][K], probs f64 [T][E])."""
    x = _f64(np.atleast_2d(x))
    T, H = x.shape
    E = router.shape[0]
    router = _f32(router)
    bias = _f32(bias)
    force = None if force is None else np.ascontiguousarray(force, dtype=np.int32)
    logits = np.empty((T, E), dtype=np.float32)
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    probs = np.empty((T, E), dtype=np.float64)
    rc = lib().qo_router(T, H, E, K, int(bool(norm_topk)), _p(x, C.c_double), _p(router, C.c_float),
                         _p(bias, C.c_float), _p(force, C.c_int32), _p(logits, C.c_float),
                         _p(ids, C.c_int32), _p(w, C.c_double), _p(probs, C.c_double))
    if rc:
        raise ValueError("router failed")
    return logits, ids, w, probs


def moe_ffn(x, ids, w, gate, up, down, gate_t, up_t, down_t, F, E, res=None, want_act=False):
    """out [T][H] (f64) = res + sum_j w_j * Wd(silu(Wg x) * Wu x); optional act [T][K][F]."""
    x = _f64(np.atleast_2d(x))
    T, H = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    K = ids.shape[1]
    w = _f64(w)
    res = None if res is None else _f64(np.atleast_2d(res))
    out = np.empty((T, H), dtype=np.float64)
    act = np.empty((T, K, F), dtype=np.float64) if want_act else None
    g8, u8, d8 = _u8(gate).reshape(-1), _u8(up).reshape(-1), _u8(down).reshape(-1)
    rc = lib().qo_moe_ffn(T, H, F, E, K, _p(x, C.c_double), _p(res, C.c_double), _p(ids, C.c_int32),
                          _p(w, C.c_double), _p(g8, C.c_uint8), QCODE[gate_t], _p(u8, C.c_uint8),
                          QCODE[up_t], _p(d8, C.c_uint8), QCODE[down_t], _p(out, C.c_double),
                          _p(act, C.c_double), None)
    if rc:
        raise ValueError(f"moe_ffn failed rc={rc}")
    return (out, act) if want_act else out


# ----------------------------------------------------------------------------- Q8_K activations

def q8k_quantize(x):
    """Q8_K blocks of a float vector (length a multiple of 256): d [n/256] (f32),
    q [n] (int8), bsums [n/16] (int16).  See qo_q8k_quantize for the reading."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    n = x.size
    d = np.empty(n // 256, dtype=np.float32)
    q = np.empty(n, dtype=np.int8)
    bs = np.empty(n // 16, dtype=np.int16)
    if lib().qo_q8k_quantize(n, _p(x, C.c_float), _p(d, C.c_float), _p(q, C.c_int8), _p(bs, C.c_int16)):
        raise ValueError("length must be a multiple of 256")
    return d, q, bs


def q8k_dot(qtype: str, row: np.ndarray, cols: int, q8) -> float:
    """One weight row (cols/256 superblocks) against Q8_K blocks, integer form."""
    d, q, bs = (np.ascontiguousarray(a) for a in q8)
    row = _u8(row).reshape(-1)
    return lib().qo_dot_q8k(QCODE[qtype], _p(row, C.c_uint8), cols, _p(d, C.c_float),
                            _p(q, C.c_int8), _p(bs, C.c_int16))


def moe_ffn_q8k(x, ids, w, gate, up, down, gate_t, up_t, down_t, F, E, res=None, want_act=False):
    """moe_ffn with every expert GEMV on Q8_K activations (x for gate/up, act for down)."""
    x = _f64(np.atleast_2d(x))
    T, H = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    K = ids.shape[1]
    w = _f64(w)
    res = None if res is None else _f64(np.atleast_2d(res))
    out = np.empty((T, H), dtype=np.float64)
    act = np.empty((T, K, F), dtype=np.float64) if want_act else None
    g8, u8, d8 = _u8(gate).reshape(-1), _u8(up).reshape(-1), _u8(down).reshape(-1)
    rc = lib().qo_moe_ffn_q8k(T, H, F, E, K, _p(x, C.c_double), _p(res, C.c_double),
                              _p(ids, C.c_int32), _p(w, C.c_double), _p(g8, C.c_uint8), QCODE[gate_t],
                              _p(u8, C.c_uint8), QCODE[up_t], _p(d8, C.c_uint8), QCODE[down_t],
                              _p(out, C.c_double), _p(act, C.c_double))
    if rc:
        raise ValueError(f"moe_ffn_q8k failed rc={rc}")
    return (out, act) if want_act else out


def moe_forward_q8k(inp: dict, norm_topk=True, force=None):
    """out = x + MoE(x) with Q8_K activations in every expert GEMV (F32 router)."""
    logits, ids, w, probs = route(inp["x"], inp["router"], inp["K"], inp.get("bias"), norm_topk,
                                  force)
    out = moe_ffn_q8k(inp["x"], ids, w, inp["gate"], inp["up"], inp["down"], inp["gate_t"],
                      inp["up_t"], inp["down_t"], inp["F"], inp["E"])
    return dict(out=out, ids=ids, w=w, logits=logits, probs=probs)


def moe_forward(inp: dict, norm_topk=True, force=None):
    """out = x + MoE(x) for one layer's synthetic inputs (see ``synth.moe_inputs``)."""
    logits, ids, w, probs = route(inp["x"], inp["router"], inp["K"], inp.get("bias"), norm_topk,
                                  force)
    out = moe_ffn(inp["x"], ids, w, inp["gate"], inp["up"], inp["down"], inp["gate_t"],
                  inp["up_t"], inp["down_t"], inp["F"], inp["E"])
    return dict(out=out, ids=ids, w=w, logits=logits, probs=probs)


# ----------------------------------------------------------------------------- FP8 experts

def fp8_e4m3_to_double(code: int) -> float:
    """Value of one E4M3 ("e4m3fn") code; NaN for S.1111.111."""
    return lib().qo_fp8_e4m3_to_double(int(code) & 0xFF)


def fp8_scale_count(rows: int, cols: int) -> int:
    """Number of fp32 block scales (one per 128 x 128 tile) of a [rows][cols] matrix."""
    return lib().qo_fp8_scale_count(rows, cols)


def fp8_dequant_matrix(codes: np.ndarray, scale: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """W[r][c] = e4m3(codes[r][c]) * scale[r // 128][c // 128], in double."""
    codes = _u8(codes).reshape(-1)
    scale = _f32(scale).reshape(-1)
    if codes.size != rows * cols or scale.size != fp8_scale_count(rows, cols):
        raise ValueError("fp8_dequant_matrix: size mismatch")
    out = np.empty((rows, cols), dtype=np.float64)
    lib().qo_fp8_dequant_matrix(_p(codes, C.c_uint8), _p(scale, C.c_float), rows, cols,
                                _p(out, C.c_double))
    return out


def moe_ffn_fp8(x, ids, w, gate, gate_scale, up, up_scale, down, down_scale, F, E, res=None,
                want_act=False):
    """out [T][H] (f64) = res + sum_j w_j * Wd(silu(Wg x) * Wu x) over FP8 block-scaled
    experts (gate/up [E][F][H] codes, down [E][H][F], fp32 scales per 128 x 128 tile)."""
    x = _f64(np.atleast_2d(x))
    T, H = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    K = ids.shape[1]
    w = _f64(w)
    res = None if res is None else _f64(np.atleast_2d(res))
    if (_u8(gate).size != E * F * H or _u8(up).size != E * F * H or _u8(down).size != E * H * F
            or _f32(gate_scale).size != E * fp8_scale_count(F, H)
            or _f32(up_scale).size != E * fp8_scale_count(F, H)
            or _f32(down_scale).size != E * fp8_scale_count(H, F)):
        raise ValueError("moe_ffn_fp8: tensor sizes do not match E, F, H")
    out = np.empty((T, H), dtype=np.float64)
    act = np.empty((T, K, F), dtype=np.float64) if want_act else None
    g8, u8, d8 = _u8(gate).reshape(-1), _u8(up).reshape(-1), _u8(down).reshape(-1)
    gs, us, ds = (_f32(a).reshape(-1) for a in (gate_scale, up_scale, down_scale))
    rc = lib().qo_moe_ffn_fp8(T, H, F, E, K, _p(x, C.c_double), _p(res, C.c_double),
                              _p(ids, C.c_int32), _p(w, C.c_double), _p(g8, C.c_uint8),
                              _p(gs, C.c_float), _p(u8, C.c_uint8), _p(us, C.c_float),
                              _p(d8, C.c_uint8), _p(ds, C.c_float), _p(out, C.c_double),
                              _p(act, C.c_double), None)
    if rc:
        raise ValueError(f"moe_ffn_fp8 failed rc={rc}")
    return (out, act) if want_act else out


def moe_forward_fp8(inp: dict, norm_topk=True, force=None):
    """out = x + MoE(x) over FP8 block-scaled experts with the F32 router (the
    full-precision router option of the atlasinference Qwen3 loader)."""
    logits, ids, w, probs = route(inp["x"], inp["router"], inp["K"], inp.get("bias"), norm_topk,
                                  force)
    out = moe_ffn_fp8(inp["x"], ids, w, inp["gate"], inp["gate_scale"], inp["up"],
                      inp["up_scale"], inp["down"], inp["down_scale"], inp["F"], inp["E"])
    return dict(out=out, ids=ids, w=w, logits=logits, probs=probs)


# ----------------------------------------------------------------------------- NVFP4 experts

def e2m1_to_double(code: int) -> float:
    """Value of one FP4 E2M1 code (low 4 bits)."""
    return lib().qo_e2m1_to_double(int(code) & 0x0F)


def nvfp4_dequant_matrix(codes, bscale, global_scale: float, rows: int, cols: int) -> np.ndarray:
    """W[r][c] = e2m1(code) * e4m3(bscale[r][c // 16]) * global, in double; codes
    [rows][cols/2] bytes with the even element in the low nibble."""
    codes = _u8(codes).reshape(-1)
    bscale = _u8(bscale).reshape(-1)
    if codes.size != rows * cols // 2 or bscale.size != rows * cols // 16 or cols % 16:
        raise ValueError("nvfp4_dequant_matrix: size mismatch")
    out = np.empty((rows, cols), dtype=np.float64)
    lib().qo_nvfp4_dequant_matrix(_p(codes, C.c_uint8), _p(bscale, C.c_uint8), float(global_scale),
                                  rows, cols, _p(out, C.c_double))
    return out


def nvfp4_quantize(x_bf16_bits: np.ndarray):
    """BF16 matrix (uint16 bit patterns [rows][cols]) -> (codes [rows][cols/2],
    bscale [rows][cols/16] E4M3 bytes, global fp32); see qo_nvfp4_quantize."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    rows, cols = x.shape
    codes = np.empty((rows, cols // 2), dtype=np.uint8)
    bs = np.empty((rows, cols // 16), dtype=np.uint8)
    g = np.empty(1, dtype=np.float32)
    if lib().qo_nvfp4_quantize(rows, cols, _p(x, C.c_uint16), _p(codes, C.c_uint8),
                               _p(bs, C.c_uint8), _p(g, C.c_float)):
        raise ValueError("nvfp4_quantize: cols must be a multiple of 16")
    return codes, bs, float(g[0])


_NV_NAMES = ("gate", "gate_bs", "gate_gs", "up", "up_bs", "up_gs", "down", "down_bs", "down_gs")


def moe_ffn_nvfp4(x, ids, w, ex: dict, F, E, res=None, want_act=False):
    """out [T][H] (f64) = res + sum_j w_j * Wd(silu(Wg x) * Wu x) over NVFP4 experts
    (ex: gate/up codes [E][F][H/2], *_bs [E][F][H/16], *_gs [E]; down [E][H][F/2],
    [E][H][F/16], [E])."""
    x = _f64(np.atleast_2d(x))
    T, H = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    K = ids.shape[1]
    w = _f64(w)
    res = None if res is None else _f64(np.atleast_2d(res))
    want = {"gate": E * F * H // 2, "gate_bs": E * F * H // 16, "gate_gs": E,
            "up": E * F * H // 2, "up_bs": E * F * H // 16, "up_gs": E,
            "down": E * H * F // 2, "down_bs": E * H * F // 16, "down_gs": E}
    arrs = []
    for n in _NV_NAMES:
        a = _f32(ex[n]).reshape(-1) if n.endswith("_gs") else _u8(ex[n]).reshape(-1)
        if a.size != want[n]:
            raise ValueError(f"moe_ffn_nvfp4: {n} has {a.size} elements, expected {want[n]}")
        arrs.append(a)
    out = np.empty((T, H), dtype=np.float64)
    act = np.empty((T, K, F), dtype=np.float64) if want_act else None
    ptrs = [_p(a, C.c_float if n.endswith("_gs") else C.c_uint8) for n, a in zip(_NV_NAMES, arrs)]
    rc = lib().qo_moe_ffn_nvfp4(T, H, F, E, K, _p(x, C.c_double), _p(res, C.c_double),
                                _p(ids, C.c_int32), _p(w, C.c_double), *ptrs,
                                _p(out, C.c_double), _p(act, C.c_double), None)
    if rc:
        raise ValueError(f"moe_ffn_nvfp4 failed rc={rc}")
    return (out, act) if want_act else out


def moe_forward_nvfp4(inp: dict, norm_topk=True, force=None):
    """out = x + MoE(x) over NVFP4 experts with the F32 router."""
    logits, ids, w, probs = route(inp["x"], inp["router"], inp["K"], inp.get("bias"), norm_topk,
                                  force)
    out = moe_ffn_nvfp4(inp["x"], ids, w, inp, inp["F"], inp["E"])
    return dict(out=out, ids=ids, w=w, logits=logits, probs=probs)


# ----------------------------------------------------------------------------- decoder layer

def rmsnorm(x, w, eps):
    x = _f64(x)
    out = np.empty_like(x)
    lib().qo_rmsnorm(x.size, _p(x, C.c_double), _p(_f32(w), C.c_float), eps, _p(out, C.c_double))
    return out


def rope_neox(v, pos, base):
    v = _f64(v).copy()
    lib().qo_rope_neox(v.size, _p(v, C.c_double), int(pos), float(base))
    return v


def attend(q, k_cache, v_cache, pos):
    """k_cache/v_cache: fp16 [ctx][hd] of one kv head."""
    q = _f64(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.float16).view(np.uint16)
    vc = np.ascontiguousarray(v_cache, dtype=np.float16).view(np.uint16)
    out = np.empty(q.size, dtype=np.float64)
    lib().qo_attend(q.size, _p(q, C.c_double), _p(kc, C.c_uint16), _p(vc, C.c_uint16), int(pos),
                    _p(out, C.c_double))
    return out


def decode_layer(geo: dict, small: dict, experts: dict, h, pos, force=None, debug=False):
    """One decoder layer on hidden h (f64 [H]).

    Returns dict(h, ids, w, logits, k_cache, v_cache[, q, att]).  The caller's
    caches are not modified: the layer writes slot ``pos`` of copies.
    """
    h = _f64(h).copy()
    kc = np.ascontiguousarray(small["k_cache"], dtype=np.float16).copy()
    vc = np.ascontiguousarray(small["v_cache"], dtype=np.float16).copy()
    K, E = geo["K"], geo["E"]
    ids = np.empty(K, dtype=np.int32)
    w = np.empty(K, dtype=np.float64)
    logits = np.empty(E, dtype=np.float32)
    force = None if force is None else np.ascontiguousarray(force, dtype=np.int32)
    args = [geo["H"], E, K, geo["F"], geo["n_heads"], geo["n_kv"], geo["head_dim"], geo["ctx"],
            geo["eps"], geo["rope_base"], int(pos), _p(h, C.c_double)]
    norms = [_f32(small[n]) for n in ("attn_norm", "q_norm", "k_norm", "ffn_norm")]
    args += [_p(a, C.c_float) for a in norms]
    keep = [_u8(small[n]).reshape(-1) for n in ("wq", "wk", "wv", "wo")]
    args += [_p(a, C.c_uint8) for a in keep]
    ex = [_u8(experts[n]).reshape(-1) for n in ("gate", "up", "down")]
    router = _f32(small["router"])
    args += [_p(router, C.c_float)] + [_p(a, C.c_uint8) for a in ex]
    args += [QCODE[small["down_t"]], _p(kc.view(np.uint16), C.c_uint16),
             _p(vc.view(np.uint16), C.c_uint16), _p(force, C.c_int32), _p(logits, C.c_float),
             _p(ids, C.c_int32), _p(w, C.c_double)]
    qd = geo["n_heads"] * geo["head_dim"]
    q = np.empty(qd, dtype=np.float64) if debug else None
    att = np.empty(qd, dtype=np.float64) if debug else None
    args += [_p(q, C.c_double), _p(att, C.c_double)]
    rc = lib().qo_decode_layer(*args)
    if rc:
        raise ValueError(f"decode_layer failed rc={rc}")
    out = dict(h=h, ids=ids, w=w, logits=logits, k_cache=kc, v_cache=vc)
    if debug:
        out.update(q=q, att=att)
    return out


def prefill_layer(geo: dict, small: dict, experts: dict, hs, pos0: int, force=None):
    """One decoder layer on T tokens at positions pos0 .. pos0+T-1 (prefill).

    Within one layer a token's K and V depend on its own input only, so causal
    attention over the cache (positions < pos0, as stored) and the earlier
    tokens of the batch is exactly the layer applied token by token, each
    writing its K/V slot before the next reads it (the token-by-token prefill
    of the aprender issue "qwen3moe ... has NO working CUDA path", later gap
    list, which a batched prefill must reproduce).  hs: f64 [T][H].  force
    (optional): [T][K] expert ids.  Returns dict(h [T][H], ids [T][K], w [T][K],
    router logits f32 [T][E], k_cache, v_cache) with the caches' slots pos0.. pos0+T-1 written (copies)."""
    hs = np.atleast_2d(_f64(hs))
    T = hs.shape[0]
    if pos0 < 0 or pos0 + T > geo["ctx"]:
        raise ValueError("prefill positions outside the context")
    cur = dict(small)
    outs, ids, ws, lgs = [], [], [], []
    for i in range(T):
        r = decode_layer(geo, cur, experts, hs[i], pos0 + i,
                         force=None if force is None else np.asarray(force)[i])
        cur = dict(cur, k_cache=r["k_cache"], v_cache=r["v_cache"])
        outs.append(r["h"])
        ids.append(r["ids"])
        ws.append(r["w"])
        lgs.append(r["logits"])
    return dict(h=np.stack(outs), ids=np.stack(ids), w=np.stack(ws), logits=np.stack(lgs),
                k_cache=cur["k_cache"], v_cache=cur["v_cache"])

