"""Shared helpers for the parity tests: seeded inputs -> (GPU decoder, CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from qwen3_prefill_kv_gb300 import synth

# The parity gate for teacher-forced logits: cosine >= 0.9995 and
# max|d| <= 1e-2 * max|oracle logit|, argmax equal wherever the oracle's
# top-1/top-2 gap exceeds that bound.
COS_MIN = 0.9995
REL_BOUND = 1e-2


def oracle_weights(w: synth.Weights) -> dict:
    f = lambda t: t.to(torch.float64).numpy()
    return {"embed": f(w.embed), "final_norm": f(w.final_norm),
            "layers": [{k: f(v) for k, v in l.items()} for l in w.layers]}


def make_oracle(w: synth.Weights) -> oracle.DecoderOracle:
    return oracle.DecoderOracle(w.shape, oracle_weights(w))


def audio_f64(p: synth.Prompt) -> np.ndarray:
    return p.audio.to(torch.float64).numpy()


def teacher_forced(dec, orc, prompt: synth.Prompt, n_steps: int, device="cuda"):
    """The oracle greedy-decodes and is the teacher; the GPU prefills the same
    prompt and is fed the oracle's token at every step ("Qwen3ASR ncnn多平台移植"
    §7.1).  Returns per-step (gpu_logits, oracle_logits, gpu_argmax) lists."""
    V = orc.V
    logits = torch.empty(V, dtype=torch.float32, device=device)
    out = []
    z_ref = orc.prefill(prompt.ids.numpy(), audio_f64(prompt), prompt.audio_offset)
    a = dec.prefill(prompt.ids, prompt.audio.to(device) if prompt.audio.numel() else None,
                    prompt.audio_offset, logits=logits)
    out.append((logits.cpu().numpy().astype(np.float64), z_ref, a))
    for _ in range(n_steps):
        tok = oracle.greedy_argmax(z_ref)
        z_ref = orc.decode_step(tok)
        a = dec.decode_step(tok, logits=logits)
        out.append((logits.cpu().numpy().astype(np.float64), z_ref, a))
    return out


def assert_step_parity(steps, label=""):
    worst = None
    for i, (g, r, a) in enumerate(steps):
        ok, m = oracle.parity_gate(g, r, COS_MIN, REL_BOUND)
        # the GPU argmax is the argmax of the GPU's own logits (lowest index on ties)
        assert a == int(np.argmax(g)), f"{label} step {i}: argmax {a} != argmax of returned logits {int(np.argmax(g))}"
        assert ok, f"{label} step {i}: parity gate failed: {m}"
        if worst is None or m["max_abs"] / m["max_abs_ref"] > worst["max_abs"] / worst["max_abs_ref"]:
            worst = dict(m, step=i)
    return worst
