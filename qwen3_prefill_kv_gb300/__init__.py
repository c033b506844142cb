"""GB300 (sm_103a) library for the Qwen3-0.6B-shape causal decoder of speech-LLM ASR
pipelines: multimodal prefill with spliced audio rows, KV-cache decode, tied lm_head
with greedy argmax, context cloning and batched lockstep decode.

``synth`` (seeded inputs) imports no compiled code; ``_lib`` loads ``libqdec.so``
lazily and raises when it is missing (there is no CPU fallback).
"""
from . import synth  # noqa: F401

__all__ = ["synth", "Decoder", "load"]


def __getattr__(name):
    if name in ("Decoder", "load", "QdecError"):
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
