"""Seeded synthetic inputs for the Qwen3-0.6B-shape decoder path.

This module is the only code shared by the CPU oracle's callers and the CUDA
path's callers.  It draws random numbers and lays them out; it holds none of
the decoder's arithmetic.

Shapes follow the model tuple (hidden 1024, ffn 3072, 28 layers, 16 q heads,
8 kv heads, head_dim 128, vocab 151936) of "Fun-ASR-Nano Native Runtime
Implementation Plan", Task 1 Step 1, and the "LLM decoder (Qwen3-0.6B, frozen,
BF16)" table of "Forward map - funasr_nano".  No checkpoint exists here, so
weights are random: every weight matrix is N(0, 0.02) rounded to bf16, norm
gains are 1 (or 1 + N(0, 0.1) with ``gain_jitter``), audio rows are
N(0, 1) * 0.5 rounded to bf16 and token ids are uniform on [0, vocab).

Recipe (stable for a given seed, independent of thread scheduling):
  * Every tensor has a fixed index in the order embed, then per layer
    (wqkv, wo, wgu, wd, g_in, g_post, g_q, g_k), then final_norm.
  * Each tensor is filled in chunks of 2**22 elements; chunk ``c`` of tensor
    ``t`` is drawn by ``torch.randn`` from a CPU Generator seeded with
    ``_chunk_seed(seed, t, c)``.
  * Prompt ids, audio rows and forced tokens come from their own Generators
    seeded with ``_stream_seed(seed, tag)``.

Weight layout (row-major ``[out, in]``, bf16):
  * ``wqkv`` [(Hq + 2*Hkv) * D, H]: rows [0, Hq*D) are q (head-major), then
    Hkv*D rows of k, then Hkv*D rows of v.
  * ``wgu`` [2F, H]: rows [0, F) are gate, rows [F, 2F) are up ("packed
    gate_up" in the forward map's decoder table).
  * ``wo`` [H, Hq*D], ``wd`` [H, F].
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, asdict
import os

import torch

_CHUNK = 1 << 22


@dataclass(frozen=True)
class ModelShape:
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def kv_bytes_per_position(self) -> int:
        """bf16 K and V of one position over all layers."""
        return self.n_layers * 2 * self.n_kv_heads * self.head_dim * 2

    def weight_params(self) -> int:
        per_layer = (self.qkv_rows * self.hidden + self.hidden * self.n_q_heads * self.head_dim
                     + 2 * self.ffn * self.hidden + self.hidden * self.ffn
                     + 2 * self.hidden + 2 * self.head_dim)
        return self.vocab * self.hidden + self.n_layers * per_layer + self.hidden

    def as_dict(self) -> dict:
        return asdict(self)


TINY = ModelShape(hidden=128, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=32,
                  ffn=384, vocab=1024)
QWEN3_06B = ModelShape(hidden=1024, n_layers=28, n_q_heads=16, n_kv_heads=8, head_dim=128,
                       ffn=3072, vocab=151936)


@dataclass(frozen=True)
class Workload:
    """One prompt layout + decode schedule.

    The prompt is ``n_prefix`` text ids, ``n_audio`` audio rows spliced at
    offset ``n_prefix``, then ``n_suffix`` text ids; ``n_decode`` decode steps
    follow at batch ``batch`` (batch > 1 means clones of one prefill state).
    """
    name: str
    shape: ModelShape
    n_prefix: int
    n_audio: int
    n_suffix: int
    n_decode: int
    batch: int = 1
    description: str = ""

    @property
    def n_prompt(self) -> int:
        return self.n_prefix + self.n_audio + self.n_suffix

    @property
    def audio_offset(self) -> int:
        return self.n_prefix

    @property
    def max_seq(self) -> int:
        return self.n_prompt + self.n_decode


WORKLOADS = {
    "tiny": Workload("tiny", TINY, 12, 8, 12, 16,
                     description="tiny Qwen3-style decoder, 32-position prompt, 16 decode steps"),
    # 23 audio rows = fake_token_len(183) ("Forward map - funasr_nano", Adaptor table).
    "funasr_nano_short": Workload("funasr_nano_short", QWEN3_06B, 20, 23, 21, 64,
                                  description="Qwen3-0.6B shape, 64-position prompt (20 ids, 23 audio rows, 21 ids), 64 decode steps"),
    "qwen3_asr_30s": Workload("qwen3_asr_30s", QWEN3_06B, 15, 390, 10, 256,
                              description="Qwen3-0.6B shape, 415-position prompt (15 ids, 390 audio rows, 10 ids), 256 decode steps"),
    "long_context": Workload("long_context", QWEN3_06B, 32, 4032, 32, 256,
                             description="Qwen3-0.6B shape, 4096-position prompt (32 ids, 4032 audio rows, 32 ids), 256 decode steps"),
    "branching_b64": Workload("branching_b64", QWEN3_06B, 15, 390, 10, 128, batch=64,
                              description="415-position prefill, 64 clones, 128 lockstep decode steps at batch 64"),
}


def _chunk_seed(seed: int, tensor_index: int, chunk: int) -> int:
    return (seed * 1_000_003 + tensor_index * 65_537 + chunk) & 0x7FFF_FFFF_FFFF


def _stream_seed(seed: int, tag: int) -> int:
    return (seed * 7_919 + 0x5EED_0000 + tag) & 0x7FFF_FFFF_FFFF


def _normal_bf16(shape, std: float, mean: float, seed: int, tensor_index: int,
                 pool: ThreadPoolExecutor) -> torch.Tensor:
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=torch.bfloat16)

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = torch.Generator().manual_seed(_chunk_seed(seed, tensor_index, c))
        v = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if mean != 0.0:
            v.add_(mean)
        out[lo:hi] = v.to(torch.bfloat16)

    list(pool.map(fill, range((n + _CHUNK - 1) // _CHUNK)))
    return out.view(*shape)


@dataclass
class Weights:
    """bf16 CPU tensors in the layout documented at the top of this module."""
    shape: ModelShape
    embed: torch.Tensor
    final_norm: torch.Tensor
    layers: list = field(default_factory=list)  # dicts: wqkv, wo, wgu, wd, g_in, g_post, g_q, g_k

    def tensors(self):
        yield "embed", self.embed
        for i, l in enumerate(self.layers):
            for k in ("wqkv", "wo", "wgu", "wd", "g_in", "g_post", "g_q", "g_k"):
                yield f"layers.{i}.{k}", l[k]
        yield "final_norm", self.final_norm

    def to(self, device) -> "Weights":
        return Weights(self.shape, self.embed.to(device), self.final_norm.to(device),
                       [{k: v.to(device) for k, v in l.items()} for l in self.layers])


def make_weights(shape: ModelShape, seed: int = 0, gain_jitter: bool = False,
                 weight_std: float = 0.02) -> Weights:
    """Random-init bf16 weights of ``shape`` (see the module docstring for the recipe)."""
    H, D, F = shape.hidden, shape.head_dim, shape.ffn
    idx = 0
    threads = min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as pool:
        def mat(rows, cols):
            nonlocal idx
            t = _normal_bf16((rows, cols), weight_std, 0.0, seed, idx, pool)
            idx += 1
            return t

        def gain(n):
            nonlocal idx
            if gain_jitter:
                t = _normal_bf16((n,), 0.1, 1.0, seed, idx, pool)
            else:
                t = torch.ones(n, dtype=torch.bfloat16)
            idx += 1
            return t

        embed = mat(shape.vocab, H)
        layers = []
        for _ in range(shape.n_layers):
            l = {}
            l["wqkv"] = mat(shape.qkv_rows, H)
            l["wo"] = mat(H, shape.n_q_heads * D)
            l["wgu"] = mat(2 * F, H)
            l["wd"] = mat(H, F)
            l["g_in"] = gain(H)
            l["g_post"] = gain(H)
            l["g_q"] = gain(D)
            l["g_k"] = gain(D)
            layers.append(l)
        final_norm = gain(H)
    return Weights(shape, embed, final_norm, layers)


@dataclass
class Prompt:
    ids: torch.Tensor       # int32 [n_prompt]; positions covered by audio hold 0
    audio: torch.Tensor     # bf16 [n_audio, hidden]
    audio_offset: int


def make_prompt(w: Workload, seed: int = 0) -> Prompt:
    g = torch.Generator().manual_seed(_stream_seed(seed, 1))
    ids = torch.randint(0, w.shape.vocab, (w.n_prompt,), generator=g, dtype=torch.int64).to(torch.int32)
    ids[w.audio_offset:w.audio_offset + w.n_audio] = 0
    ga = torch.Generator().manual_seed(_stream_seed(seed, 2))
    audio = (torch.randn(w.n_audio, w.shape.hidden, generator=ga) * 0.5).to(torch.bfloat16)
    return Prompt(ids, audio, w.audio_offset)


def make_tokens(vocab: int, n: int, seed: int = 0, tag: int = 3) -> torch.Tensor:
    """``n`` token ids uniform on [0, vocab) (forced first tokens of clones, etc.)."""
    g = torch.Generator().manual_seed(_stream_seed(seed, tag))
    return torch.randint(0, vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32)


# ------------------------------------------------------------------ audio adaptor inputs
@dataclass(frozen=True)
class AdaptorShape:
    """The projector and bidirectional adaptor that turn encoder frames into the audio rows
    spliced into the prompt ("Forward map - funasr_nano", adaptor table: linear1 512 -> 2048
    + ReLU, linear2 2048 -> 1024, two blocks of LayerNorm + multi-head attention + a
    1024 -> 256 -> 1024 ReLU FFN; "Fun-ASR-Nano Native Runtime Implementation Plan", Task 5:
    eight heads)."""
    enc_dim: int = 512
    proj_dim: int = 2048
    hidden: int = 1024
    n_heads: int = 8
    ffn: int = 256
    n_blocks: int = 2
    ln_eps: float = 1.0e-12


ADAPTOR = AdaptorShape()
ADAPTOR_TINY = AdaptorShape(enc_dim=24, proj_dim=40, hidden=32, n_heads=4, ffn=8, n_blocks=2)


def make_adaptor_weights(shape: AdaptorShape, seed: int = 0, weight_std: float = 0.02) -> dict:
    """Random-init float32 adaptor weights: matrices N(0, weight_std), biases N(0, 0.02),
    LayerNorm gains 1 + N(0, 0.1) and biases N(0, 0.1) (non-trivial, so a dropped affine
    term shows), drawn from one Generator seeded with _stream_seed(seed, 16) in the order
    listed; matrices row-major [out, in]."""
    g = torch.Generator().manual_seed(_stream_seed(seed, 16))

    def mat(o, i):
        return torch.randn(o, i, generator=g) * weight_std

    def vec(n, std, mean=0.0):
        return torch.randn(n, generator=g) * std + mean

    E, P, H, F = shape.enc_dim, shape.proj_dim, shape.hidden, shape.ffn
    w = {"w1": mat(P, E), "b1": vec(P, 0.02), "w2": mat(H, P), "b2": vec(H, 0.02), "blocks": []}
    for _ in range(shape.n_blocks):
        w["blocks"].append({
            "ln1_g": vec(H, 0.1, 1.0), "ln1_b": vec(H, 0.1),
            "wq": mat(H, H), "bq": vec(H, 0.02), "wk": mat(H, H), "bk": vec(H, 0.02),
            "wv": mat(H, H), "bv": vec(H, 0.02), "wo": mat(H, H), "bo": vec(H, 0.02),
            "ln2_g": vec(H, 0.1, 1.0), "ln2_b": vec(H, 0.1),
            "fc1": mat(F, H), "fc1_b": vec(F, 0.02), "fc2": mat(H, F), "fc2_b": vec(H, 0.02)})
    return w


def make_encoder_frames(shape: AdaptorShape, n_frames: int, seed: int = 0) -> torch.Tensor:
    """Encoder output frames [n_frames, enc_dim], N(0, 1) float32."""
    g = torch.Generator().manual_seed(_stream_seed(seed, 17))
    return torch.randn(n_frames, shape.enc_dim, generator=g)
