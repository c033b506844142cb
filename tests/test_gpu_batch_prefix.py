"""Shared-prefix attention of the lockstep batch ("Qwen3ASR ncnn多平台移植" §5: clones of one
prefill state decode as branches).  Clones of one prefill hold the same keys and values at
the prompt positions, so the batch attends that prefix once, from one member's cache, for
every member's queries.  Checked against the oracle's clones, against the same batch with
the sharing switched off, and on compositions that mix prefixes."""
import numpy as np
import pytest
import torch

import oracle
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Decoder

import _harness as H

pytestmark = pytest.mark.gpu

# head_dim 128 (what the shared-prefix kernel covers) at a small width: 4 q heads over 2 kv
# heads, 2 layers, vocabulary 1024
SH128 = synth.ModelShape(hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=512, vocab=1024)


@pytest.fixture(scope="module")
def model():
    w = synth.make_weights(SH128, seed=0)
    return w, w.to("cuda"), H.make_oracle(w)


def _prompt(n_prefix, n_audio, n_suffix, seed=0):
    return synth.make_prompt(synth.Workload("t", SH128, n_prefix, n_audio, n_suffix, 0), seed)


def _branches(src, n):
    return [src.clone() for _ in range(n)]


@pytest.mark.parametrize("layout,n", [((10, 50, 10), 5), ((3, 30, 4), 70), ((1, 0, 0), 3), ((20, 60, 17), 2)])
def test_shared_prefix_matches_oracle_and_private_attention(model, layout, n):
    """n clones stepped 4 times: every stream against its oracle clone, and against the same
    composition with QDEC_OPT_SHARED_PREFIX = 0 (each stream over its own copy).  70 streams
    overflow one block of query rows (64 streams of 2 heads); prompts of 1, 41, 70 and 97
    positions give prefixes shorter than one 32-key chunk, ragged chunks and several chunks."""
    w, wd, orc = model
    p = _prompt(*layout)
    T = p.ids.numel()
    src = Decoder(SH128, wd, max_seq=T + 8)
    src.prefill(p.ids, p.audio.cuda() if p.audio.numel() else None, p.audio_offset)
    o_src = orc.clone()
    o_src.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    shared = _branches(src, n)
    private = _branches(src, n)
    private[0].set_option(_lib.OPT_SHARED_PREFIX, 0)
    assert shared[0].get_option(_lib.OPT_SHARED_PREFIX) == 1
    obr = [o_src.clone() for _ in range(n)]
    toks = synth.make_tokens(SH128.vocab, n, seed=11).numpy()
    la = torch.empty(n, SH128.vocab, device="cuda")
    lb = torch.empty(n, SH128.vocab, device="cuda")
    for step in range(4):
        am = Decoder.decode_step_batch(shared, toks, logits=la)
        Decoder.decode_step_batch(private, toks, logits=lb)
        ga, gb = la.cpu().numpy(), lb.cpu().numpy()
        assert np.array_equal(am, ga.argmax(axis=1))
        for i in range(n):
            z = obr[i].decode_step(int(toks[i]))
            ok, m = oracle.parity_gate(ga[i], z, H.COS_MIN, H.REL_BOUND)
            assert ok, (step, i, m)
            # both read the same bf16 cache; the prefix part rounds q and the probabilities to
            # bf16 for its tensor-core products
            np.testing.assert_allclose(ga[i], gb[i], rtol=0, atol=1e-2 * float(np.abs(gb[i]).max()),
                                       err_msg=f"step {step} stream {i}")
        toks = am
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32)
    for i in (0, n - 1):   # the caches themselves: the prefix untouched, the new slots written per stream
        ks, kp = shared[i].read_kv(1, 0, 0, T + 4), private[i].read_kv(1, 0, 0, T + 4)
        assert np.array_equal(ks[:, :T], kp[:, :T])
        np.testing.assert_allclose(f(ks[:, T:]), f(kp[:, T:]), rtol=0, atol=2e-2 * float(np.abs(f(kp)).max()))


def test_mixed_prefixes_in_one_batch(model):
    """Clones of two different prefills, interleaved, plus one context with a prompt of its own:
    two groups share their own prefixes, the singleton attends over its copy."""
    w, wd, orc = model
    pa, pb, pc = _prompt(6, 20, 6, seed=1), _prompt(4, 40, 9, seed=2), _prompt(5, 10, 5, seed=3)
    srcs, osrcs = [], []
    for p in (pa, pb, pc):
        d = Decoder(SH128, wd, max_seq=64)
        d.prefill(p.ids, p.audio.cuda(), p.audio_offset)
        o = orc.clone()
        o.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
        srcs.append(d)
        osrcs.append(o)
    order = [0, 1, 0, 1, 0, 2, 1]
    batch = [srcs[k].clone() for k in order]
    obr = [osrcs[k].clone() for k in order]
    n = len(batch)
    toks = synth.make_tokens(SH128.vocab, n, seed=4).numpy()
    lg = torch.empty(n, SH128.vocab, device="cuda")
    for step in range(3):
        am = Decoder.decode_step_batch(batch, toks, logits=lg)
        g = lg.cpu().numpy()
        for i in range(n):
            ok, m = oracle.parity_gate(g[i], obr[i].decode_step(int(toks[i])), H.COS_MIN, H.REL_BOUND)
            assert ok, (step, i, m)
        toks = am
    # a re-prefilled member leaves its group: the next step must rebuild the groups
    batch[2].prefill(pa.ids, pa.audio.cuda(), pa.audio_offset)
    obr[2] = orc.clone()
    obr[2].prefill(pa.ids.numpy(), H.audio_f64(pa), pa.audio_offset)
    am = Decoder.decode_step_batch(batch, toks, logits=lg)
    g = lg.cpu().numpy()
    for i in range(n):
        ok, m = oracle.parity_gate(g[i], obr[i].decode_step(int(toks[i])), H.COS_MIN, H.REL_BOUND)
        assert ok, ("after re-prefill", i, m)


def test_shared_prefix_option_validation(model):
    w, wd, orc = model
    d = Decoder(SH128, wd, max_seq=16)
    with pytest.raises(_lib.QdecError):
        d.set_option(_lib.OPT_SHARED_PREFIX, 2)
    d.set_option(_lib.OPT_SHARED_PREFIX, 0)
    assert d.clone().get_option(_lib.OPT_SHARED_PREFIX) == 0
