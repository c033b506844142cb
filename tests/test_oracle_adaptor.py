"""Pins of the adaptor oracle (oracle/adaptor.py): the projector + two-block bidirectional
adaptor of "Forward map - funasr_nano" (section "Adaptor"), against closed forms, brute
force, library routines (torch layer_norm, scaled_dot_product_attention, linear, relu) and
planted mistakes that the independent formulation must catch."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from oracle import adaptor as A
from qwen3_prefill_kv_gb300 import synth

SH = synth.ADAPTOR_TINY


def _w(seed=0):
    w = synth.make_adaptor_weights(SH, seed=seed, weight_std=0.3)
    f = lambda t: t.double().numpy()
    return {"w1": f(w["w1"]), "b1": f(w["b1"]), "w2": f(w["w2"]), "b2": f(w["b2"]),
            "blocks": [{k: f(v) for k, v in b.items()} for b in w["blocks"]]}


def _torch_adaptor(frames, w, heads, eps, causal=False, post_norm=False, proj_relu=True, rms=False):
    """Independent formulation from library routines (the planted-mistake switches flip one
    reading each)."""
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    x = Fn.linear(T(frames), T(w["w1"]), T(w["b1"]))
    x = Fn.relu(x) if proj_relu else x
    x = Fn.linear(x, T(w["w2"]), T(w["b2"]))

    def norm(v, g, b):
        if rms:
            return v * torch.rsqrt((v * v).mean(-1, keepdim=True) + eps) * T(g) + T(b)
        return Fn.layer_norm(v, (v.shape[-1],), T(g), T(b), eps)

    for b in w["blocks"]:
        n, H = x.shape
        d = H // heads
        def attn(v):
            q = Fn.linear(v, T(b["wq"]), T(b["bq"])).view(n, heads, d).transpose(0, 1)
            k = Fn.linear(v, T(b["wk"]), T(b["bk"])).view(n, heads, d).transpose(0, 1)
            vv = Fn.linear(v, T(b["wv"]), T(b["bv"])).view(n, heads, d).transpose(0, 1)
            o = Fn.scaled_dot_product_attention(q, k, vv, is_causal=causal)
            return Fn.linear(o.transpose(0, 1).reshape(n, H), T(b["wo"]), T(b["bo"]))
        def ffn(v):
            return Fn.linear(Fn.relu(Fn.linear(v, T(b["fc1"]), T(b["fc1_b"]))), T(b["fc2"]), T(b["fc2_b"]))
        if post_norm:
            x = norm(x + attn(x), b["ln1_g"], b["ln1_b"])
            x = norm(x + ffn(x), b["ln2_g"], b["ln2_b"])
        else:
            x = x + attn(norm(x, b["ln1_g"], b["ln1_b"]))
            x = x + ffn(norm(x, b["ln2_g"], b["ln2_b"]))
    return x.numpy()


def test_layer_norm_closed_form_and_library():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, 32)) * 3 + 1
    g, b = rng.normal(size=32), rng.normal(size=32)
    y = A.layer_norm(x, np.ones(32), np.zeros(32), 1e-12)
    np.testing.assert_allclose(y.mean(-1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(-1), 1.0, rtol=1e-10)
    ref = Fn.layer_norm(torch.from_numpy(x), (32,), torch.from_numpy(g), torch.from_numpy(b), 1e-12).numpy()
    np.testing.assert_allclose(A.layer_norm(x, g, b, 1e-12), ref, rtol=1e-12, atol=1e-12)


def test_mha_brute_force_on_a_tiny_clip():
    rng = np.random.default_rng(1)
    T, H, heads = 3, 4, 2
    d = H // heads
    blk = {k: rng.normal(size=(H, H)) for k in ("wq", "wk", "wv", "wo")}
    blk.update({k: rng.normal(size=H) for k in ("bq", "bk", "bv", "bo")})
    x = rng.normal(size=(T, H))
    proj = lambda w, b: [[sum(x[t][i] * w[o][i] for i in range(H)) + b[o] for o in range(H)] for t in range(T)]
    q, k, v = proj(blk["wq"], blk["bq"]), proj(blk["wk"], blk["bk"]), proj(blk["wv"], blk["bv"])
    cat = [[0.0] * H for _ in range(T)]
    for h in range(heads):
        for t in range(T):
            sc = [sum(q[t][h * d + e] * k[j][h * d + e] for e in range(d)) / math.sqrt(d) for j in range(T)]
            mx = max(sc)
            ex = [math.exp(s - mx) for s in sc]
            for e in range(d):
                cat[t][h * d + e] = sum(ex[j] * v[j][h * d + e] for j in range(T)) / sum(ex)
    out = [[sum(cat[t][i] * blk["wo"][o][i] for i in range(H)) + blk["bo"][o] for o in range(H)] for t in range(T)]
    np.testing.assert_allclose(A.bidirectional_mha(x, blk, heads), np.array(out), rtol=1e-12, atol=1e-12)


def test_mha_is_permutation_equivariant_and_single_frame_is_value_path():
    w = _w()
    blk = w["blocks"][0]
    rng = np.random.default_rng(2)
    x = rng.normal(size=(9, SH.hidden))
    perm = rng.permutation(9)
    np.testing.assert_allclose(A.bidirectional_mha(x[perm], blk, SH.n_heads),
                               A.bidirectional_mha(x, blk, SH.n_heads)[perm], rtol=1e-12, atol=1e-12)
    one = x[:1]
    expect = A.linear(A.linear(one, blk["wv"], blk["bv"]), blk["wo"], blk["bo"])
    np.testing.assert_allclose(A.bidirectional_mha(one, blk, SH.n_heads), expect, rtol=1e-12, atol=1e-12)


def test_whole_adaptor_matches_library_formulation():
    w = _w()
    frames = synth.make_encoder_frames(SH, 17, seed=3).double().numpy()
    got = A.adaptor(frames, w, SH.n_heads, SH.ln_eps)
    ref = _torch_adaptor(frames, w, SH.n_heads, SH.ln_eps)
    assert np.abs(got - ref).max() <= 1e-10 * np.abs(ref).max()


@pytest.mark.parametrize("mistake", ["causal", "post_norm", "no_proj_relu", "rms", "eps"])
def test_planted_mistakes_are_caught(mistake):
    w = _w()
    frames = synth.make_encoder_frames(SH, 17, seed=3).double().numpy()
    got = A.adaptor(frames, w, SH.n_heads, SH.ln_eps)
    kw = {"causal": dict(causal=True), "post_norm": dict(post_norm=True), "no_proj_relu": dict(proj_relu=False),
          "rms": dict(rms=True), "eps": {}}[mistake]
    eps = 1e-5 if mistake == "eps" else SH.ln_eps
    bad = _torch_adaptor(frames, w, SH.n_heads, eps, **kw)
    assert np.abs(got - bad).max() > 1e-8 * np.abs(bad).max()


def test_audio_rows_take_fake_token_len_rows():
    w = _w()
    frames = synth.make_encoder_frames(SH, 183, seed=4).double().numpy()
    rows = A.audio_rows(frames, w, SH.n_heads, SH.ln_eps)
    assert rows.shape == (23, SH.hidden)   # the page's 183 frames -> 23 rows
    np.testing.assert_array_equal(rows, A.adaptor(frames, w, SH.n_heads, SH.ln_eps)[:23])


def test_full_shape_generators():
    w = synth.make_adaptor_weights(synth.ADAPTOR, seed=0)
    assert tuple(w["w1"].shape) == (2048, 512) and tuple(w["w2"].shape) == (1024, 2048)
    b = w["blocks"][1]
    assert tuple(b["fc1"].shape) == (256, 1024) and tuple(b["fc2"].shape) == (1024, 256)
    assert len(w["blocks"]) == 2 and synth.ADAPTOR.n_heads == 8 and synth.ADAPTOR.ln_eps == 1e-12
    again = synth.make_adaptor_weights(synth.ADAPTOR, seed=0)
    assert torch.equal(w["w1"], again["w1"]) and torch.equal(b["fc2_b"], again["blocks"][1]["fc2_b"])
