"""CPU oracle for the Qwen3-0.6B-shape causal decoder hot path.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` are the only code that may import
or run anything in this package.  The CUDA library and its Python binding never
import, link or call it, and this package imports nothing from them: callers
hand it plain arrays (the seeded inputs) and compare its results with the GPU's.

Every function computes in float64 (see ``decoder.py`` for the reading of the
pages this follows).  Parity is pinned by ``tests/test_oracle_pins.py``.
``sampling.py`` is the token choice after the lm_head (greedy, temperature, top-k,
top-p, repetition penalty, counter-based draws), pinned by
``tests/test_oracle_sampling.py``; ``adaptor.py`` is the projector and bidirectional
adaptor that produce the audio rows, pinned by ``tests/test_oracle_adaptor.py``;
``quant.py`` is the library's block-quantized weight formats, pinned by
``tests/test_oracle_quant.py``.
"""
from .decoder import (DecoderOracle, rms_norm, rope_inv_freq, rope_neox, causal_gqa_attention,
                      swiglu, inputs_embeds, tied_lm_head, greedy_argmax, fake_token_len)
from .metrics import step_metrics, parity_gate

__all__ = ["DecoderOracle", "rms_norm", "rope_inv_freq", "rope_neox", "causal_gqa_attention",
           "swiglu", "inputs_embeds", "tied_lm_head", "greedy_argmax", "fake_token_len",
           "step_metrics", "parity_gate"]
