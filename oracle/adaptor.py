"""Float64 reference of the projector and bidirectional adaptor that produce the audio rows
spliced into the decoder's prompt.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code imports it.

What it follows: "Forward map - funasr_nano", section "Adaptor (Transformer, n_layer=2,
downsample_rate=1, use_low_frame_rate=true)": an identity reshape (k = 1), linear1
512 -> 2048 with bias and ReLU, linear2 2048 -> 1024 with bias, then two blocks, each
norm1 -> q/k/v/out projections with biases -> residual, norm2 -> fc1 1024 -> 256 + ReLU +
fc2 256 -> 1024 with biases -> residual, where the norms are LayerNorm with bias and
eps 1e-12 and the attention is plain (no Q/K norm, no RoPE); then the host keeps the first
fake_token_len rows for the splice.  "Fun-ASR-Nano Native Runtime Implementation Plan",
Task 5: eight-head bidirectional attention, pre-norm blocks, residuals.

Readings where the pages are silent: attention over all frames of the clip (bidirectional,
no mask within one clip), scaled by 1/sqrt(head_dim), heads contiguous in the projection
rows; no norm after the last block (the table lists none); LayerNorm uses the population
variance.
"""
from __future__ import annotations

import math

import numpy as np

from .decoder import fake_token_len


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def layer_norm(x, g, b, eps: float) -> np.ndarray:
    """(x - mean) / sqrt(var + eps) * g + b over the last axis (population variance)."""
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * _f64(g) + _f64(b)


def linear(x, w, b) -> np.ndarray:
    """x @ w^T + b with w row-major [out, in]."""
    return _f64(x) @ _f64(w).T + _f64(b)


def bidirectional_mha(x, blk, n_heads: int) -> np.ndarray:
    """Multi-head attention of every frame over every frame of the clip: softmax(q k^T /
    sqrt(d)) v per head, heads concatenated, then the output projection."""
    T, H = x.shape
    d = H // n_heads
    q = linear(x, blk["wq"], blk["bq"]).reshape(T, n_heads, d)
    k = linear(x, blk["wk"], blk["bk"]).reshape(T, n_heads, d)
    v = linear(x, blk["wv"], blk["bv"]).reshape(T, n_heads, d)
    out = np.empty((T, n_heads, d))
    for h in range(n_heads):
        s = q[:, h, :] @ k[:, h, :].T / math.sqrt(d)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, h, :]
    return linear(out.reshape(T, H), blk["wo"], blk["bo"])


def adaptor_block(x, blk, n_heads: int, eps: float) -> np.ndarray:
    """One pre-norm block: x + MHA(LN1(x)), then + fc2(ReLU(fc1(LN2(.))))."""
    x = _f64(x)
    x = x + bidirectional_mha(layer_norm(x, blk["ln1_g"], blk["ln1_b"], eps), blk, n_heads)
    hdn = np.maximum(linear(layer_norm(x, blk["ln2_g"], blk["ln2_b"], eps), blk["fc1"], blk["fc1_b"]), 0.0)
    return x + linear(hdn, blk["fc2"], blk["fc2_b"])


def adaptor(frames, w, n_heads: int, eps: float) -> np.ndarray:
    """Encoder frames [T, 512] -> adaptor output [T, 1024] (projector, then the blocks)."""
    x = linear(np.maximum(linear(frames, w["w1"], w["b1"]), 0.0), w["w2"], w["b2"])
    for blk in w["blocks"]:
        x = adaptor_block(x, blk, n_heads, eps)
    return x


def audio_rows(frames, w, n_heads: int, eps: float) -> np.ndarray:
    """The rows spliced into the prompt: the first fake_token_len(T) adaptor outputs."""
    out = adaptor(frames, w, n_heads, eps)
    return out[:fake_token_len(out.shape[0])]
