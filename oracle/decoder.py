"""Float64 reference of the Qwen3 causal decoder that the pages' ASR pipelines share.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code imports it.

What it follows:
  * "Forward map - funasr_nano", table "LLM decoder (Qwen3-0.6B, frozen, BF16)":
    token embedding by row gather, audio rows overriding ``inputs_embeds`` at
    ``[fbank_beg, fbank_beg + fake_token_len)``, 28 pre-norm blocks of
    rms_norm + GQA 16/8 + per-head Q/K RMSNorm + NeoX RoPE (theta 1e6) + SwiGLU
    (packed gate_up), a final RMSNorm and the tied lm_head on the last position.
  * Same page, table "Generation / KV Path": prefill writes the KV cache for
    [0, T_prompt); each later step runs one token at n_past >= T_prompt.
  * "Qwen3ASR ncnn多平台移植", section 4 (audio-pad rows of the text embedding are
    replaced by audio embeddings, so positions and modality order match the
    Torch forward) and section 5 (prefill with an upper-triangular causal mask,
    28-layer KV cache, logits of the last prompt position; each decode step
    embeds one token, builds RoPE for its absolute position, attends over the
    whole history plus itself, appends its K/V and runs the LM head; the
    context keeps KV, history and position and can be cloned to branch).
  * "Fun-ASR-Nano Native Runtime Implementation Plan", Task 1 Step 1 (the shape
    tuple and theta 1e6) and Task 6 Step 5 (prefill logits, greedy steps and
    KV-cache parity as the decoder's checks).

Readings where the pages are silent (each is listed in the design notes):
  * q rows of the packed projection are 16 x 128 = 2048 wide, k and v 8 x 128;
    o_proj maps 2048 -> 1024; no biases anywhere in the block.
  * Q/K RMSNorm comes before RoPE (the order the decoder table lists them).
  * NeoX pairs are (i, i + D/2) with inverse frequency theta^(-2i/D).
  * q head h reads kv head h // (Hq / Hkv).
  * Packed gate_up: rows [0, F) gate, [F, 2F) up.
  * Audio rows replace (not add to) the embedded rows; ids under them are ignored.
  * The lm_head is evaluated on the last prompt position only; argmax takes
    the lowest index among equal maxima.

Precision: float64 everywhere, cache included.  The pages compare a float32
CPU port against a bfloat16 Torch model and fix no single precision, so the
oracle computes the exact function of the bf16 weights.
"""
from __future__ import annotations

import math
from typing import Mapping, Sequence

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def rms_norm(x, gain, eps: float) -> np.ndarray:
    """x / sqrt(mean(x**2) + eps) * gain over the last axis.

    The decoder table's ``rms_norm`` (before attention and before the MLP), the
    per-head Q/K RMSNorm (over each head's D values) and ``model.norm`` before
    the head ("Forward map - funasr_nano", "LLM decoder" table)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(gain)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2i/D) for i in [0, D/2): one frequency per rotated pair."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_neox(x, positions, theta: float) -> np.ndarray:
    """NeoX ("rotate-half") rotary embedding at absolute positions.

    x is [T, heads, D]; element i < D/2 is paired with i + D/2 and the pair is
    rotated by the angle position * theta^(-2i/D) ("NeoX RoPE @ 1e6" in the
    decoder table of "Forward map - funasr_nano"; the RoPE cos/sin cache of
    "Qwen3ASR ncnn多平台移植", section 5 step 2)."""
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    ang = _f64(positions)[:, None] * rope_inv_freq(d, theta)[None, :]      # [T, D/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def causal_gqa_attention(q, k, v, q_pos, k_pos) -> np.ndarray:
    """Grouped-query attention with a causal mask.

    q [T, Hq, D]; k, v [L, Hkv, D].  Query t (absolute position q_pos[t]) sees
    key j iff k_pos[j] <= q_pos[t] (the upper-triangular causal mask of
    "Qwen3ASR ncnn多平台移植" section 5; a decode step's single-row mask covers
    the history and itself).  Scores are q.k / sqrt(D); softmax subtracts the
    row maximum.  q head h reads kv head h // (Hq / Hkv) ("GQA 16/8")."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, d = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    visible = _f64(k_pos)[None, :] <= _f64(q_pos)[:, None]                 # [T, L]
    out = np.empty((T, hq, d), dtype=np.float64)
    scale = 1.0 / math.sqrt(d)
    for h in range(hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def swiglu(gate_up, ffn: int) -> np.ndarray:
    """silu(gate) * up for a packed [.., 2F] projection (gate first, then up);
    silu(z) = z / (1 + exp(-z)).  "SwiGLU (packed gate_up)" in the decoder table."""
    gu = _f64(gate_up)
    g, u = gu[..., :ffn], gu[..., ffn:]
    return g / (1.0 + np.exp(-g)) * u


def inputs_embeds(embed, ids, audio, audio_offset: int) -> np.ndarray:
    """Row gather of the token embedding, then the audio rows override
    positions [audio_offset, audio_offset + n_audio).

    "Forward map - funasr_nano", decoder table rows "Token embed"
    (``ggml_get_rows``) and "Audio-row override" (``inputs_embeds[...,
    fbank_beg:fbank_beg+L] = adaptor_out[:L]``); "Qwen3ASR ncnn多平台移植"
    section 4 (audio_pad rows replaced by audio embeddings)."""
    e = np.asarray(embed)
    ids = np.asarray(ids, dtype=np.int64)
    x = _f64(e[ids])
    if audio is not None and len(audio) > 0:
        a = _f64(audio)
        x[audio_offset:audio_offset + a.shape[0]] = a
    return x


def tied_lm_head(embed, h) -> np.ndarray:
    """logits = E . h with the token embedding as the output matrix ("Tied
    lm_head" in the decoder table; ``mul_mat(token_w, last_x)``)."""
    return _f64(embed) @ _f64(h)


def greedy_argmax(logits) -> int:
    """Index of the largest logit, lowest index on ties (greedy decode,
    temperature 0: "Qwen3ASR ncnn多平台移植" section 6 default config).
    A NaN is an error."""
    z = _f64(logits)
    if np.isnan(z).any():
        raise FloatingPointError("NaN in logits")
    return int(np.argmax(z))


def fake_token_len(n_frames: int) -> int:
    """Number of adaptor frames spliced into the prompt (host arithmetic).

    "Forward map - funasr_nano", Adaptor table: three nested ``(n-1)/2 + 1``
    stages; the page's worked example is 183 frames -> 23.  The formula as
    printed there ends in ``/2+1`` and would give 24 for 183; the reading that
    reproduces the page's own example applies the same ``(n-1)//2 + 1``
    halving three times."""
    n = int(n_frames)
    for _ in range(3):
        n = (n - 1) // 2 + 1
    return n


class DecoderOracle:
    """Prefill / decode / clone over a float64 KV cache.

    ``shape`` is a mapping or object with hidden, n_layers, n_q_heads,
    n_kv_heads, head_dim, ffn, vocab, rope_theta, rms_eps.  ``weights`` has
    ``embed`` [V, H], ``final_norm`` [H] and ``layers``: a list of mappings with
    wqkv [(Hq+2Hkv)D, H], wo [H, Hq D], wgu [2F, H], wd [H, F], g_in [H],
    g_post [H], g_q [D], g_k [D].  Arrays are widened to float64 once."""

    def __init__(self, shape, weights):
        get = (lambda k: shape[k]) if isinstance(shape, Mapping) else (lambda k: getattr(shape, k))
        self.H = int(get("hidden"))
        self.NL = int(get("n_layers"))
        self.HQ = int(get("n_q_heads"))
        self.HKV = int(get("n_kv_heads"))
        self.D = int(get("head_dim"))
        self.F = int(get("ffn"))
        self.V = int(get("vocab"))
        self.theta = float(get("rope_theta"))
        self.eps = float(get("rms_eps"))
        wget = (lambda k: weights[k]) if isinstance(weights, Mapping) else (lambda k: getattr(weights, k))
        self.embed = _f64(wget("embed"))
        self.final_norm = _f64(wget("final_norm"))
        self.layers = [{k: _f64(v) for k, v in l.items()} for l in wget("layers")]
        self.reset()

    # -- state ---------------------------------------------------------------
    def reset(self) -> None:
        self.k_cache = [np.zeros((0, self.HKV, self.D)) for _ in range(self.NL)]
        self.v_cache = [np.zeros((0, self.HKV, self.D)) for _ in range(self.NL)]
        self.history: list[int] = []
        self.position = 0

    def clone(self) -> "DecoderOracle":
        """Independent copy of the context: KV cache, history, position
        ("Qwen3ASR ncnn多平台移植" section 5: generate() clones its input context
        so several branches can start from one prefill state).  Weights are shared."""
        c = object.__new__(DecoderOracle)
        c.__dict__.update({k: v for k, v in self.__dict__.items()
                           if k not in ("k_cache", "v_cache", "history")})
        c.k_cache = [k.copy() for k in self.k_cache]
        c.v_cache = [v.copy() for v in self.v_cache]
        c.history = list(self.history)
        return c

    # -- one pre-norm block ----------------------------------------------------
    def _block(self, l: int, x: np.ndarray, positions: np.ndarray) -> np.ndarray:
        w = self.layers[l]
        hq, hkv, d = self.HQ, self.HKV, self.D
        t = x.shape[0]
        xn = rms_norm(x, w["g_in"], self.eps)
        qkv = xn @ w["wqkv"].T
        q = qkv[:, :hq * d].reshape(t, hq, d)
        k = qkv[:, hq * d:(hq + hkv) * d].reshape(t, hkv, d)
        v = qkv[:, (hq + hkv) * d:].reshape(t, hkv, d)
        q = rope_neox(rms_norm(q, w["g_q"], self.eps), positions, self.theta)
        k = rope_neox(rms_norm(k, w["g_k"], self.eps), positions, self.theta)
        # KV cache append: slot index = absolute position.
        self.k_cache[l] = np.concatenate([self.k_cache[l], k], axis=0)
        self.v_cache[l] = np.concatenate([self.v_cache[l], v], axis=0)
        k_pos = np.arange(self.k_cache[l].shape[0])
        o = causal_gqa_attention(q, self.k_cache[l], self.v_cache[l], positions, k_pos)
        x = x + o.reshape(t, hq * d) @ w["wo"].T
        xn = rms_norm(x, w["g_post"], self.eps)
        x = x + swiglu(xn @ w["wgu"].T, self.F) @ w["wd"].T
        return x

    def _forward(self, x: np.ndarray) -> np.ndarray:
        positions = np.arange(self.position, self.position + x.shape[0])
        for l in range(self.NL):
            x = self._block(l, x, positions)
        self.position += x.shape[0]
        return x

    def final_hidden(self, x_last) -> np.ndarray:
        return rms_norm(x_last, self.final_norm, self.eps)

    # -- public steps ------------------------------------------------------------
    def prefill(self, ids: Sequence[int], audio=None, audio_offset: int = 0) -> np.ndarray:
        """Runs the whole prompt from position 0 (the cache is reset), returns the
        logits of the last prompt position."""
        ids = np.asarray(ids, dtype=np.int64)
        if ids.size == 0:
            raise ValueError("empty prompt")
        n_audio = 0 if audio is None else len(audio)
        if audio_offset < 0 or audio_offset + n_audio > ids.size:
            raise ValueError("audio rows out of range")
        if (ids < 0).any() or (ids >= self.V).any():
            raise ValueError("token id out of range")
        self.reset()
        x = self._forward(inputs_embeds(self.embed, ids, audio, audio_offset))
        self.history = [int(i) for i in ids]
        return tied_lm_head(self.embed, self.final_hidden(x[-1]))

    def decode_step(self, token: int) -> np.ndarray:
        """One token at position n_past, attending over the cache plus itself."""
        if self.position == 0:
            raise RuntimeError("decode before prefill")
        token = int(token)
        if not 0 <= token < self.V:
            raise ValueError("token id out of range")
        x = self._forward(self.embed[[token]].copy())
        self.history.append(token)
        return tied_lm_head(self.embed, self.final_hidden(x[-1]))

    def full_recompute(self, ids: Sequence[int], audio=None, audio_offset: int = 0) -> np.ndarray:
        """Logits of the last position of ``ids`` from one uncached pass over the
        whole sequence (a fresh context; this one is left untouched)."""
        c = self.clone()
        return c.prefill(ids, audio, audio_offset)
