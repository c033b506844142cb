"""The allocation-free lm_head + argmax entry point.

Callers that own all device memory through their own pool, or that run on a real-time
thread where cudaMalloc's device-wide synchronisation is not acceptable, use
qdec_op_lm_head_argmax_static.  Its scratch is a library-owned static device array.
These tests call it through the C ABI and compare it with qdec_op_lm_head_argmax (which
takes caller-provided scratch) on two calls in a row: the second call checks that what
the first call left in the shared array does not leak into the result.  This file is
named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from qwen3_prefill_kv_gb300 import _lib

pytestmark = pytest.mark.gpu


def _inputs(V, H, seed):
    g = torch.Generator().manual_seed(seed)
    E = (torch.randn(V, H, generator=g) * 0.02).to(torch.bfloat16).cuda()
    x = (torch.randn(H, generator=g) * 3).cuda()
    gf = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16).cuda()
    return E, x, gf


@pytest.mark.parametrize("V,H", [(151936, 1024), (1024, 128)])
def test_static_matches_scratch_entry_point_twice(V, H):
    scratch = torch.zeros(_lib.lm_head_scratch_bytes(V), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((11, 12)):
        E, x, gf = _inputs(V, H, seed)
        ref_logits = torch.empty(V, device="cuda")
        ref_am = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        _lib.lm_head_argmax(E, V, H, x, gf, 1e-6, ref_logits, ref_am, scratch)
        logits = torch.empty(V, device="cuda")
        am = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        _lib.lm_head_argmax_static(E, V, H, x, gf, 1e-6, logits, am)
        torch.cuda.synchronize()
        ref = ref_logits.cpu().double().numpy()
        got = logits.cpu().double().numpy()
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max(), f"call {call}: logits differ"
        assert int(am.item()) == int(ref_am.item()) == int(np.argmax(got)), f"call {call}: argmax differs"
        # and against the float64 oracle on the same bf16 inputs (final RMSNorm, then E . h)
        f64 = lambda t: t.cpu().to(torch.float64).numpy()
        z = oracle.tied_lm_head(f64(E), oracle.rms_norm(f64(x), f64(gf), 1e-6))
        assert np.abs(got - z).max() <= 1e-4 * np.abs(z).max(), f"call {call}: logits differ from the oracle"


def test_static_serialised_calls_on_two_streams():
    """Calls on different streams share the one static array; ordered by an event, a call on a
    second stream still starts from a cleared ticket and gives the oracle's logits and argmax."""
    V, H = 151936, 1024
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    prev = torch.cuda.current_stream()
    for k, st in enumerate((s1, s2, s1)):
        E, x, gf = _inputs(V, H, 20 + k)
        logits = torch.empty(V, device="cuda")
        am = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        st.wait_stream(torch.cuda.current_stream())   # the inputs are written
        st.wait_stream(prev)                          # the previous call is done with the array
        _lib.lm_head_argmax_static(E, V, H, x, gf, 1e-6, logits, am, stream=st)
        prev = st
        outs.append((E, x, gf, logits, am, st))
    torch.cuda.synchronize()
    for k, (E, x, gf, logits, am, st) in enumerate(outs):
        f64 = lambda t: t.cpu().to(torch.float64).numpy()
        z = oracle.tied_lm_head(f64(E), oracle.rms_norm(f64(x), f64(gf), 1e-6))
        got = logits.cpu().double().numpy()
        assert np.abs(got - z).max() <= 1e-4 * np.abs(z).max(), k
        assert int(am.item()) == int(np.argmax(got)), k


def test_static_rejects_vocab_beyond_maximum():
    V, H = _lib.LM_HEAD_STATIC_MAX_VOCAB + 1, 8
    E = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(H, device="cuda")
    gf = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty(1, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.QdecError) as e:
        _lib.lm_head_argmax_static(E, V, H, x, gf, 1e-6, logits, am)
    assert e.value.status == -1
    assert b"exceeds" in _lib.load().qdec_last_error()
