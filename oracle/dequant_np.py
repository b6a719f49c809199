"""Second, independent k-quant dequantiser in numpy (test infrastructure only).

Written separately from ``qmoe_oracle.c`` (array reshapes instead of per-element
index arithmetic) so that the two can pin each other: they must agree bit for
bit.  fp16 fields are decoded with numpy's own float16 type.

Block formats: the public GGUF k-quant layout; the aprender issue "qwen3moe
(Qwen3-30B-A3B, Qwen3-Coder-30B-A3B, Q4_K_M) has NO working CUDA path",
section "File facts", fixes the sizes (Q4_K 144 B and Q6_K 210 B per 256
weights).
"""
from __future__ import annotations

import numpy as np


def _f16(b2: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(b2).view(np.float16).astype(np.float64).reshape(-1)


def q4k_blocks(raw: np.ndarray) -> np.ndarray:
    """raw uint8 [nb][144] -> float64 [nb][256]."""
    raw = np.asarray(raw, dtype=np.uint8).reshape(-1, 144)
    nb = raw.shape[0]
    d = _f16(raw[:, 0:2])
    dmin = _f16(raw[:, 2:4])
    sc = raw[:, 4:16].astype(np.int64)
    # 6-bit scales / mins of sub-blocks 0..7
    lo_s = sc[:, 0:4] & 63
    lo_m = sc[:, 4:8] & 63
    hi_s = (sc[:, 8:12] & 15) | ((sc[:, 0:4] >> 6) << 4)
    hi_m = (sc[:, 8:12] >> 4) | ((sc[:, 4:8] >> 6) << 4)
    s = np.concatenate([lo_s, hi_s], axis=1)          # [nb][8]
    m = np.concatenate([lo_m, hi_m], axis=1)
    qs = raw[:, 16:144].reshape(nb, 4, 32).astype(np.int64)
    q = np.stack([qs & 15, qs >> 4], axis=2).reshape(nb, 8, 32)   # sub-block 2c, 2c+1
    val = d[:, None, None] * s[:, :, None] * q - dmin[:, None, None] * m[:, :, None]
    return val.reshape(nb, 256)


def q6k_blocks(raw: np.ndarray) -> np.ndarray:
    """raw uint8 [nb][210] -> float64 [nb][256]."""
    raw = np.asarray(raw, dtype=np.uint8).reshape(-1, 210)
    nb = raw.shape[0]
    ql = raw[:, 0:128].reshape(nb, 2, 2, 32).astype(np.int64)     # [half][first/second 32][l]
    qh = raw[:, 128:192].reshape(nb, 2, 32).astype(np.int64)      # [half][l]
    sc = raw[:, 192:208].view(np.int8).astype(np.int64).reshape(nb, 2, 8)
    d = _f16(raw[:, 208:210])
    low = np.stack([ql[:, :, 0] & 15, ql[:, :, 1] & 15, ql[:, :, 0] >> 4, ql[:, :, 1] >> 4],
                   axis=2)                                         # [nb][half][group][l]
    high = np.stack([(qh >> (2 * g)) & 3 for g in range(4)], axis=2)
    q = (low | (high << 4)) - 32
    l16 = np.arange(32) // 16                                      # scale index within a group
    scale = np.stack([sc[:, :, 2 * g + l16] for g in range(4)], axis=2)   # [nb][half][group][l]
    val = d[:, None, None, None] * scale * q
    return val.reshape(nb, 256)


def dequant(qtype: str, raw: np.ndarray, rows: int, cols: int) -> np.ndarray:
    fn = q4k_blocks if qtype == "Q4_K" else q6k_blocks
    return fn(raw).reshape(rows, cols)
