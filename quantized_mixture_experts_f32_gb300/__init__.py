"""GB300 (sm_103a) qwen3moe MoE FFN over GGUF k-quant experts -- Python binding.

A thin ctypes layer over the C ABI in ``include/qmoe.h`` (library
``_build/libqmoe.so``, built by ``build.py``).  It only marshals arguments:
every step of the MoE FFN runs in the library's CUDA kernels.  Tensors are
passed as raw device pointers; PyTorch is used by callers for device memory
and streams only.

Importing this package loads the library and fails loudly if it has not been
built: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqmoe.so")

QMOE_OK = 0
STATUS_NAMES = {0: "QMOE_OK", 1: "QMOE_ERR_INVALID_ARG", 2: "QMOE_ERR_MISALIGNED",
                3: "QMOE_ERR_UNSUPPORTED_QTYPE", 4: "QMOE_ERR_SHAPE", 5: "QMOE_ERR_NO_MEMORY",
                6: "QMOE_ERR_CUDA", 7: "QMOE_ERR_TIMEOUT", 8: "QMOE_ERR_DEVICE_CHECK"}
QMOE_Q4_K, QMOE_Q6_K = 1, 2
QTYPE = {"Q4_K": QMOE_Q4_K, "Q6_K": QMOE_Q6_K}

# kernels one qmoe_forward enqueues on the decode path (n_tokens <= 8): the
# whole layer is one kernel (the batch-1 kernel for one token, the fused
# cooperative kernel for 2..8)
LAUNCHES_PER_DECODE_FORWARD = 1
# n_tokens > 8 (tensor-core path): router GEMM, top-k, per-expert lists, gather,
# gate/up GEMM, down GEMM, combine
LAUNCHES_PER_PREFILL_FORWARD = 7
# qmoe_forward_q8k up to 8 tokens: routing (one launch), quantise x, gate/up,
# quantise act, down, combine (7 beyond 8 tokens: router and top-k apart)
LAUNCHES_PER_Q8K_FORWARD = 6
# qmoe_forward_fp8 up to 32 tokens: routing (one launch up to 8 tokens, router
# + top-k beyond), gate/up GEMV, down GEMV, combine; more than 32 tokens (tensor
# cores): router GEMM, top-k, per-expert lists, gather, gate/up GEMM, down GEMM,
# combine
FP8_GEMV_MAX = 32
# one token at hidden 2048 / ffn 768 (up to 128 experts): the whole FP8 or NVFP4
# layer is one kernel
LAUNCHES_PER_LOWBIT_T1 = 1
LAUNCHES_PER_FP8_FORWARD = 4           # otherwise up to 8 tokens (5 for 9..32)
LAUNCHES_PER_FP8_FORWARD_MANY = 7
# qmoe_forward_nvfp4: as qmoe_forward_fp8 (4 launches up to 8 tokens, 5 for
# 9..32, 7 on the tensor cores beyond)
LAUNCHES_PER_NVFP4_FORWARD = 4
# one decoder layer of qmoe_decode_step: RMSNorm + Q/K/V GEMV, attention (with
# Q/K norm, RoPE and the KV append), split merge, O GEMV, fused MoE layer (with
# its RMSNorm)
LAUNCHES_PER_DECODE_LAYER = 5
# plus, once per qmoe_decode_step: the RoPE cos/sin table at the step's position
LAUNCHES_PER_DECODE_STEP = 1
# one decoder layer of qmoe_prefill up to the MoE input: RMSNorm, one Q/K/V
# GEMM, RoPE cos/sin table, Q/K norm + RoPE + KV append, attention, O GEMM, FFN
# RMSNorm (with the O projection's residual); the MoE adds
# LAUNCHES_PER_PREFILL_FORWARD (n_tokens > 8) or one fused kernel
LAUNCHES_PER_PREFILL_LAYER_ATTN = 7

EXPORTED = ["qmoe_create", "qmoe_destroy", "qmoe_set_stream", "qmoe_forward", "qmoe_forward_ex",
            "qmoe_forward_host", "qmoe_decode_step", "qmoe_prefill", "qmoe_get_status", "qmoe_last_error",
            "qmoe_workspace_bytes", "qmoe_expert_stride", "qmoe_forward_noalloc",
            "qmoe_fused_decode_available", "qmoe_forward_q8k", "qmoe_forward_fp8", "qmoe_forward_nvfp4",
            "qmoe_nvfp4_quantize", "qmoe_noalloc_status",
            "qmoe_debug_stall_next", "qmoe_debug_fail_alloc"]


class qmoe_config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_experts", C.c_int), ("top_k", C.c_int),
                ("ffn", C.c_int), ("norm_topk_prob", C.c_int), ("max_tokens", C.c_int),
                ("n_heads", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int),
                ("max_ctx", C.c_int), ("rope_base", C.c_float), ("rms_eps", C.c_float),
                ("stream", C.c_void_p)]


class qmoe_layer_weights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("wq", C.c_void_p), ("wk", C.c_void_p),
                ("wv", C.c_void_p), ("wo", C.c_void_p), ("q_norm", C.c_void_p),
                ("k_norm", C.c_void_p), ("ffn_norm", C.c_void_p), ("router_w", C.c_void_p),
                ("gate_exps", C.c_void_p), ("up_exps", C.c_void_p), ("down_exps", C.c_void_p),
                ("down_t", C.c_int), ("k_cache", C.c_void_p), ("v_cache", C.c_void_p)]


class QmoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libqmoe is not built ({LIB_PATH} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` -- there is no CPU fallback")
    L = C.CDLL(LIB_PATH)
    vp, i, ip, fp = C.c_void_p, C.c_int, C.c_void_p, C.c_void_p
    L.qmoe_create.argtypes = [C.POINTER(qmoe_config), C.POINTER(C.c_void_p)]
    L.qmoe_create.restype = i
    L.qmoe_destroy.argtypes = [vp]
    L.qmoe_destroy.restype = None
    L.qmoe_set_stream.argtypes = [vp, vp]
    L.qmoe_set_stream.restype = i
    L.qmoe_forward.argtypes = [vp, fp, fp, vp, vp, vp, i, i, i, i, fp]
    L.qmoe_forward.restype = i
    L.qmoe_forward_ex.argtypes = [vp, fp, fp, fp, fp, vp, vp, vp, i, i, i, i, fp, ip, fp]
    L.qmoe_forward_ex.restype = i
    L.qmoe_forward_host.argtypes = [vp, fp, fp, vp, vp, vp, i, i, i, i, fp]
    L.qmoe_forward_q8k.argtypes = [vp, fp, fp, vp, vp, vp, i, i, i, i, fp, ip, fp]
    L.qmoe_forward_q8k.restype = i
    L.qmoe_forward_fp8.argtypes = [vp, fp, fp, vp, fp, vp, fp, vp, fp, i, fp, ip, fp]
    L.qmoe_forward_fp8.restype = i
    L.qmoe_forward_nvfp4.argtypes = [vp, fp, fp] + [vp, vp, fp] * 3 + [i, fp, ip, fp]
    L.qmoe_forward_nvfp4.restype = i
    L.qmoe_nvfp4_quantize.argtypes = [vp, vp, i, i, i, vp, vp, fp]
    L.qmoe_nvfp4_quantize.restype = i
    L.qmoe_forward_host.restype = i
    L.qmoe_decode_step.argtypes = [vp, C.POINTER(qmoe_layer_weights), i, i, fp, ip]
    L.qmoe_decode_step.restype = i
    L.qmoe_prefill.argtypes = [vp, C.POINTER(qmoe_layer_weights), i, i, i, fp, ip]
    L.qmoe_prefill.restype = i
    L.qmoe_get_status.argtypes = [vp]
    L.qmoe_get_status.restype = i
    L.qmoe_last_error.argtypes = [vp]
    L.qmoe_last_error.restype = C.c_char_p
    L.qmoe_workspace_bytes.argtypes = [C.POINTER(qmoe_config)]
    L.qmoe_workspace_bytes.restype = C.c_size_t
    L.qmoe_fused_decode_available.argtypes = [vp, i, i, i, i]
    L.qmoe_fused_decode_available.restype = i
    L.qmoe_expert_stride.argtypes = [i, i, i]
    L.qmoe_expert_stride.restype = C.c_size_t
    L.qmoe_forward_noalloc.argtypes = [fp, fp, vp, vp, vp, i, i, i, i, i, i, i, i, i, fp, vp]
    L.qmoe_forward_noalloc.restype = i
    L.qmoe_noalloc_status.argtypes = [vp]
    L.qmoe_noalloc_status.restype = i
    L.qmoe_debug_stall_next.argtypes = [vp, C.c_uint64]
    L.qmoe_debug_stall_next.restype = i
    L.qmoe_debug_fail_alloc.argtypes = [i]
    L.qmoe_debug_fail_alloc.restype = None
    return L


lib = _load()


def _ptr(t):
    """Device (or host) address of a tensor-like object, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _check(ctx, status):
    if status != QMOE_OK:
        msg = lib.qmoe_last_error(ctx).decode() if ctx else ""
        raise QmoeError(status, msg)


# ---------------------------------------------------------------------------- C names

def qmoe_create(cfg: qmoe_config):
    h = C.c_void_p()
    st = lib.qmoe_create(C.byref(cfg), C.byref(h))
    if st != QMOE_OK:
        raise QmoeError(st, lib.qmoe_last_error(None).decode())
    return h


def qmoe_destroy(ctx):
    lib.qmoe_destroy(ctx)


def qmoe_set_stream(ctx, stream: int):
    _check(ctx, lib.qmoe_set_stream(ctx, stream))


def qmoe_forward(ctx, hidden_in, router_w, gate_exps, up_exps, down_exps, gate_t, up_t, down_t,
                 n_tokens, hidden_out):
    _check(ctx, lib.qmoe_forward(ctx, _ptr(hidden_in), _ptr(router_w), _ptr(gate_exps),
                                 _ptr(up_exps), _ptr(down_exps), gate_t, up_t, down_t, n_tokens,
                                 _ptr(hidden_out)))


def qmoe_forward_ex(ctx, ffn_in, residual, router_bias, router_w, gate_exps, up_exps, down_exps,
                    gate_t, up_t, down_t, n_tokens, out, ids_out=None, weights_out=None):
    _check(ctx, lib.qmoe_forward_ex(ctx, _ptr(ffn_in), _ptr(residual), _ptr(router_bias),
                                    _ptr(router_w), _ptr(gate_exps), _ptr(up_exps),
                                    _ptr(down_exps), gate_t, up_t, down_t, n_tokens, _ptr(out),
                                    _ptr(ids_out), _ptr(weights_out)))


def qmoe_forward_q8k(ctx, hidden_in, router_w, gate_exps, up_exps, down_exps, gate_t, up_t, down_t,
                     n_tokens, hidden_out, ids_out=None, weights_out=None):
    _check(ctx, lib.qmoe_forward_q8k(ctx, _ptr(hidden_in), _ptr(router_w), _ptr(gate_exps),
                                     _ptr(up_exps), _ptr(down_exps), gate_t, up_t, down_t,
                                     n_tokens, _ptr(hidden_out), _ptr(ids_out), _ptr(weights_out)))


def qmoe_forward_fp8(ctx, hidden_in, router_w, gate_exps, gate_scale, up_exps, up_scale,
                     down_exps, down_scale, n_tokens, hidden_out, ids_out=None, weights_out=None):
    _check(ctx, lib.qmoe_forward_fp8(ctx, _ptr(hidden_in), _ptr(router_w), _ptr(gate_exps),
                                     _ptr(gate_scale), _ptr(up_exps), _ptr(up_scale),
                                     _ptr(down_exps), _ptr(down_scale), n_tokens,
                                     _ptr(hidden_out), _ptr(ids_out), _ptr(weights_out)))


def qmoe_forward_nvfp4(ctx, hidden_in, router_w, gate_exps, gate_bscale, gate_global, up_exps,
                       up_bscale, up_global, down_exps, down_bscale, down_global, n_tokens,
                       hidden_out, ids_out=None, weights_out=None):
    _check(ctx, lib.qmoe_forward_nvfp4(ctx, _ptr(hidden_in), _ptr(router_w), _ptr(gate_exps),
                                       _ptr(gate_bscale), _ptr(gate_global), _ptr(up_exps),
                                       _ptr(up_bscale), _ptr(up_global), _ptr(down_exps),
                                       _ptr(down_bscale), _ptr(down_global), n_tokens,
                                       _ptr(hidden_out), _ptr(ids_out), _ptr(weights_out)))


def qmoe_nvfp4_quantize(ctx, x_bf16, n_mats, rows, cols, codes, bscale, global_scale):
    _check(ctx, lib.qmoe_nvfp4_quantize(ctx, _ptr(x_bf16), n_mats, rows, cols, _ptr(codes),
                                        _ptr(bscale), _ptr(global_scale)))


def qmoe_forward_host(ctx, hidden_in_host, router_w, gate_exps, up_exps, down_exps, gate_t, up_t,
                      down_t, n_tokens, hidden_out_host):
    _check(ctx, lib.qmoe_forward_host(ctx, _ptr(hidden_in_host), _ptr(router_w), _ptr(gate_exps),
                                      _ptr(up_exps), _ptr(down_exps), gate_t, up_t, down_t,
                                      n_tokens, _ptr(hidden_out_host)))


def qmoe_decode_step(ctx, layers, n_layers, pos, hidden, ids_out=None):
    _check(ctx, lib.qmoe_decode_step(ctx, layers, n_layers, pos, _ptr(hidden), _ptr(ids_out)))


def qmoe_prefill(ctx, layers, n_layers, n_tokens, pos0, hidden, ids_out=None):
    _check(ctx, lib.qmoe_prefill(ctx, layers, n_layers, n_tokens, pos0, _ptr(hidden), _ptr(ids_out)))


def qmoe_forward_noalloc(hidden_in, router_w, gate_exps, up_exps, down_exps, gate_t, up_t,
                         down_t, hidden, n_experts, top_k, ffn, norm_topk_prob, n_tokens,
                         hidden_out, stream=0) -> int:
    """Allocation-free decode-size forward; returns the qmoe_status code."""
    return lib.qmoe_forward_noalloc(_ptr(hidden_in), _ptr(router_w), _ptr(gate_exps),
                                    _ptr(up_exps), _ptr(down_exps), gate_t, up_t, down_t, hidden,
                                    n_experts, top_k, ffn, norm_topk_prob, n_tokens,
                                    _ptr(hidden_out), stream or None)


def qmoe_noalloc_status(stream=0) -> int:
    """Device status of the last qmoe_forward_noalloc call on this device (clears it)."""
    return lib.qmoe_noalloc_status(stream or None)


def qmoe_debug_stall_next(ctx, wait_ns: int):
    _check(ctx, lib.qmoe_debug_stall_next(ctx, wait_ns))


def qmoe_debug_fail_alloc(n: int):
    lib.qmoe_debug_fail_alloc(n)


def qmoe_get_status(ctx) -> int:
    return lib.qmoe_get_status(ctx)


def qmoe_last_error(ctx) -> str:
    return lib.qmoe_last_error(ctx).decode()


def qmoe_workspace_bytes(cfg: qmoe_config) -> int:
    return lib.qmoe_workspace_bytes(C.byref(cfg))


def qmoe_fused_decode_available(ctx, n_tokens: int, gate_t: int, up_t: int, down_t: int) -> bool:
    return bool(lib.qmoe_fused_decode_available(ctx, n_tokens, gate_t, up_t, down_t))


def qmoe_expert_stride(qtype: int, rows: int, cols: int) -> int:
    return lib.qmoe_expert_stride(qtype, rows, cols)


def make_config(hidden, n_experts, top_k, ffn, max_tokens, norm_topk_prob=1, stream=0,
                n_heads=0, n_kv_heads=0, head_dim=0, max_ctx=0, rope_base=0.0,
                rms_eps=0.0) -> qmoe_config:
    return qmoe_config(hidden, n_experts, top_k, ffn, norm_topk_prob, max_tokens, n_heads,
                       n_kv_heads, head_dim, max_ctx, rope_base, rms_eps, stream or None)
