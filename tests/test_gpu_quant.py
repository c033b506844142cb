"""Quantized-weight decode (QDEC_OPT_WEIGHTS: the library's q8b32 and q4b32 block formats;
"Fun-ASR-Nano Native Runtime Implementation Plan", Task 8).  The device quantizer must give
the oracle's codes and scales bit for bit; the quantized GEMV must match a float64 product
with the dequantized weights; and a decoder whose decode steps run on quantized layer
weights must pass the parity gate against the float64 decoder oracle run on the
dequantized weights (its prefill, embedding and lm_head stay bf16)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import quant as Q
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Decoder, QdecError

import _harness as H

pytestmark = pytest.mark.gpu
FMTS = {"q8b32": _lib.WEIGHTS_Q8B32, "q4b32": _lib.WEIGHTS_Q4B32}


def _weights(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N, K, generator=g) * 0.02
    w[3] = 0.0                                              # an all-zero row: scale 0, codes 0
    w[5, :32] = torch.arange(-16, 16) * 2.0 ** -7           # a block whose values are multiples of its step
    w[7, 32:64] = 1e-30                                     # a block below fp16's range: scale rounds to 0
    return w.to(torch.bfloat16)


def _gpu_quantize(wb, fmt):
    N, K = wb.shape
    codes = torch.empty(N, K if fmt == "q8b32" else K // 2, dtype=torch.int8 if fmt == "q8b32" else torch.uint8,
                        device="cuda")
    scales = torch.empty(N, K // 32, dtype=torch.float16, device="cuda")
    _lib.quantize(wb.cuda(), N, K, FMTS[fmt], codes, scales)
    torch.cuda.synchronize()
    return codes, scales


@pytest.mark.parametrize("fmt", ["q8b32", "q4b32"])
def test_quantizer_is_bit_exact(fmt):
    wb = _weights(300, 1024, seed=1)
    codes, scales = _gpu_quantize(wb, fmt)
    q_ref, d_ref = Q.quantize(wb.to(torch.float64).numpy(), fmt)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint16), d_ref.view(np.uint16))
    got = codes.cpu().numpy()
    if fmt == "q8b32":
        np.testing.assert_array_equal(got, q_ref)
    else:
        np.testing.assert_array_equal(got, Q.pack_q4(q_ref))
        np.testing.assert_array_equal(Q.unpack_q4(got), q_ref)


@pytest.mark.parametrize("fmt", ["q8b32", "q4b32"])
@pytest.mark.parametrize("mode,norm", [(0, True), (1, False), (2, True)])
def test_quantized_gemv_matches_dequantized_product(fmt, mode, norm):
    rows, K = 200, 1024
    n_w = 2 * rows if mode == 2 else rows
    wb = _weights(n_w, K, seed=2)
    codes, scales = _gpu_quantize(wb, fmt)
    q_ref, d_ref = Q.quantize(wb.to(torch.float64).numpy(), fmt)
    wd = Q.dequantize(q_ref, d_ref)
    g = torch.Generator().manual_seed(3)
    x = torch.randn(K, generator=g) * 2.0
    gain = (1 + 0.1 * torch.randn(K, generator=g)).to(torch.bfloat16)
    y0 = torch.randn(rows, generator=g)
    y = y0.clone().cuda()
    _lib.gemv_q(codes, scales, FMTS[fmt], rows, K, x.cuda(), gain.cuda() if norm else None, 1e-6, mode, y,
                up_off=rows)
    torch.cuda.synchronize()
    xh = x.double().numpy()
    if norm:
        xh = oracle.rms_norm(xh, gain.double().numpy(), 1e-6)
    z = wd @ xh
    if mode == 0:
        ref = z
    elif mode == 1:
        ref = y0.double().numpy() + z
    else:
        ref = oracle.swiglu(z[None, :], rows)[0]
    got = y.cpu().double().numpy()
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()


SH256 = synth.ModelShape(hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=512, vocab=1024)


def _dequantized_oracle_layers(orc, w, fmt):
    """The oracle's layer matrices replaced by their dequantized float64 values."""
    for l, layer in enumerate(w.layers):
        for k in ("wqkv", "wo", "wgu", "wd"):
            q, d = Q.quantize(layer[k].to(torch.float64).numpy(), fmt)
            orc.layers[l][k] = Q.dequantize(q, d)


@pytest.mark.parametrize("fmt", ["q8b32", "q4b32"])
@pytest.mark.parametrize("shape", ["small", "qwen3_06b"])
def test_quantized_decode_matches_oracle(fmt, shape):
    sh = SH256 if shape == "small" else synth.QWEN3_06B
    wl = synth.Workload("t", sh, 20, 23, 21, 0)
    w = synth.make_weights(sh, seed=0)
    orc = H.make_oracle(w)
    p = synth.make_prompt(wl, seed=0)
    steps = 6 if shape == "small" else 3
    dec = Decoder(sh, w.to("cuda"), max_seq=wl.n_prompt + steps)
    lg = torch.empty(sh.vocab, device="cuda")
    z = orc.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    dec.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=lg)
    dec.set_option(_lib.OPT_WEIGHTS, FMTS[fmt])
    assert dec.get_option(_lib.OPT_WEIGHTS) == FMTS[fmt]
    assert dec.decode_kernel == _lib.DECODE_GRAPH
    _dequantized_oracle_layers(orc, w, fmt)
    for step in range(steps):
        tok = oracle.greedy_argmax(z)
        z = orc.decode_step(tok)
        a = dec.decode_step(tok, logits=lg)
        got = lg.cpu().double().numpy()
        ok, m = oracle.parity_gate(got, z, H.COS_MIN, H.REL_BOUND)
        assert ok, (step, m)
        assert a == int(got.argmax())
    # a clone shares the quantized copy; the persistent kernel is refused while quantized
    c = dec.clone()
    assert c.get_option(_lib.OPT_WEIGHTS) == FMTS[fmt]
    with pytest.raises(QdecError):
        c.decode_kernel = _lib.DECODE_PERSISTENT
    with pytest.raises(QdecError):
        Decoder.decode_step_batch([dec, c], [1, 2])
    dec.set_option(_lib.OPT_WEIGHTS, _lib.WEIGHTS_BF16)
    assert dec.decode_kernel == _lib.DECODE_PERSISTENT


def test_weight_format_validation():
    w = synth.make_weights(synth.TINY, seed=0).to("cuda")
    d = Decoder(synth.TINY, w, max_seq=16)
    with pytest.raises(QdecError):
        d.set_option(_lib.OPT_WEIGHTS, 3)
    with pytest.raises(QdecError):   # hidden 128: not a multiple of 256
        d.set_option(_lib.OPT_WEIGHTS, _lib.WEIGHTS_Q8B32)
