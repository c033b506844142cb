"""Reference of the block-quantized weight formats for a bandwidth-reduced decode.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code imports it.

"Fun-ASR-Nano Native Runtime Implementation Plan", Task 8, packages the decoder as F16,
Q8_0 and Q4_K_M GGUF files and compares their transcripts and logit drift, but it does not
define the block formats.  This module defines the library's own two formats, each over
blocks of 32 consecutive weights of one row (along K, the dot-product axis):

  * q8b32: one fp16 scale d = max|w| / 127 per block and 32 int8 codes
    q = clamp(round_half_even(w / d), -127, 127); w' = q * d (34 bytes per 32 weights,
    1.0625 bytes per weight against 2 for bf16);
  * q4b32: one fp16 scale d = max|w| / 7 per block and 32 signed 4-bit codes
    q = clamp(round_half_even(w / d), -7, 7), stored as q + 8 in a nibble, the lower
    nibble first; w' = q * d (18 bytes per 32 weights, 0.5625 bytes per weight).

An all-zero block has d = 0 and codes 0.  The scale is rounded to fp16 before the codes are
computed, so decoding uses exactly the stored scale.  A decoder with quantized weights is
the float64 decoder oracle run on the dequantized weights w'.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
QMAX = {"q8b32": 127, "q4b32": 7}


def quantize(w, fmt: str):
    """Rows of w [N, K] (K % 32 == 0) -> (codes int8 [N, K], scales float16 [N, K / 32])."""
    w = np.asarray(w, dtype=np.float64)
    N, K = w.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    qmax = QMAX[fmt]
    blocks = w.reshape(N, K // BLOCK, BLOCK)
    d = (np.abs(blocks).max(axis=2) / qmax).astype(np.float16)
    d64 = d.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d64 > 0, np.round(blocks / np.where(d64 > 0, d64, 1.0)), 0.0)
    q = np.clip(q, -qmax, qmax).astype(np.int8)
    return q.reshape(N, K), d


def dequantize(codes, scales) -> np.ndarray:
    """w' = code * scale of its block, float64 [N, K]."""
    codes = np.asarray(codes, dtype=np.float64)
    N, K = codes.shape
    d = np.asarray(scales, dtype=np.float64)
    return (codes.reshape(N, K // BLOCK, BLOCK) * d[..., None]).reshape(N, K)


def pack_q4(codes) -> np.ndarray:
    """4-bit codes [N, K] in [-7, 7] -> bytes [N, K / 2]: (q + 8) in nibbles, lower first."""
    u = (np.asarray(codes, dtype=np.int16) + 8).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack_q4(packed) -> np.ndarray:
    """Inverse of pack_q4."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0x0F).astype(np.int16) - 8
    hi = (p >> 4).astype(np.int16) - 8
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def bytes_per_weight(fmt: str) -> float:
    """Storage of one weight including its share of the block scale."""
    return {"q8b32": (32 + 2) / 32, "q4b32": (16 + 2) / 32}[fmt]
