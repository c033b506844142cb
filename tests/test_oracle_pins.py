"""Pins for the CPU oracle: each checks it against something other than itself.

What pins what:
  * RMSNorm: closed form on constant rows, the RMS of its output, torch's
    library ``rms_norm``.
  * NeoX RoPE: identity at position 0, pair-span (NeoX vs interleaved pairing),
    norm preservation, group law R_a R_b = R_{a+b}, relative-position property,
    complex-multiplication formulation, closed-form angle of the first pair.
  * Attention: brute-force pure-Python loops, torch's library SDPA, rows of the
    softmax summing to 1, causality under perturbation of future keys, a single
    visible key, GQA reducing to MHA with repeated kv heads.
  * SwiGLU: silu's closed forms and torch's library silu; gate/up order.
  * Splice, tied head, argmax: exact row replacement, brute-force dot products,
    lowest index on ties.
  * Whole decoder: splicing the embedding rows equals the text-only prompt,
    incremental decode equals full recompute (the KV-cache parity of the
    Fun-ASR-Nano plan, Task 6 Step 5), clone then decode equals decode, and an
    independent float64 torch formulation built on library routines.
  * fake_token_len: the page's worked example (tests/golden/fake_token_len.txt).
  * Planted mistakes (in the oracle, on the CPU) must fail the independent check.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
from oracle import decoder as od
from qwen3_prefill_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row_closed_form():
    for c in (0.5, -3.0, 1e-3):
        x = np.full((1, 64), c)
        y = oracle.rms_norm(x, np.ones(64), 1e-6)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rmsnorm_output_rms_and_gain():
    x = rng.normal(size=(5, 96))
    g = rng.normal(size=96)
    y1 = oracle.rms_norm(x, np.ones(96), 1e-6)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y1 * y1, axis=1)), np.sqrt(ms / (ms + 1e-6)), rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-6), y1 * g, rtol=1e-13)


def test_rmsnorm_matches_torch_library():
    x = rng.normal(size=(7, 128))
    g = rng.normal(size=128)
    ref = Fn.rms_norm(torch.from_numpy(x), (128,), weight=torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- RoPE
D = 32


def test_rope_identity_at_position_zero():
    x = rng.normal(size=(1, 3, D))
    assert np.array_equal(oracle.rope_neox(x, np.array([0]), 1e6), x)


def test_rope_neox_pairs_i_with_i_plus_half():
    for i in (0, 5, D // 2 - 1):
        x = np.zeros((1, 1, D))
        x[0, 0, i] = 0.7
        x[0, 0, i + D // 2] = -0.2
        y = oracle.rope_neox(x, np.array([17]), 1e6)
        others = np.delete(y[0, 0], [i, i + D // 2])
        assert np.abs(others).max() == 0.0
        assert abs(np.hypot(y[0, 0, i], y[0, 0, i + D // 2]) - np.hypot(0.7, 0.2)) < 1e-14


def test_rope_first_pair_turns_by_position_radians():
    # inverse frequency of pair 0 is theta^0 = 1, so e_0 rotates by p radians
    for p in (1, 3, 100):
        x = np.zeros((1, 1, D)); x[0, 0, 0] = 1.0
        y = oracle.rope_neox(x, np.array([p]), 1e6)[0, 0]
        np.testing.assert_allclose([y[0], y[D // 2]], [math.cos(p), math.sin(p)], atol=1e-13)


def test_rope_group_law_and_norm():
    x = rng.normal(size=(1, 2, D))
    a, b = 37, 1201
    ra = oracle.rope_neox(oracle.rope_neox(x, np.array([b]), 1e6), np.array([a]), 1e6)
    rab = oracle.rope_neox(x, np.array([a + b]), 1e6)
    np.testing.assert_allclose(ra, rab, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(rab, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_relative_position_property():
    q = rng.normal(size=(1, 1, D)); k = rng.normal(size=(1, 1, D))
    def dot(m, n):
        return float(np.sum(oracle.rope_neox(q, np.array([m]), 1e6) * oracle.rope_neox(k, np.array([n]), 1e6)))
    for m, n, s in ((5, 2, 100), (400, 17, 3000), (0, 9, 4000)):
        assert abs(dot(m, n) - dot(m + s, n + s)) < 1e-10


def test_rope_matches_complex_rotation():
    x = rng.normal(size=(4, 3, D))
    pos = np.array([0, 1, 415, 4351])
    half = D // 2
    omega = np.exp(-np.log(1e6) * (2.0 * np.arange(half) / D))
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * pos[:, None, None] * omega[None, None, :])
    ref = np.concatenate([z.real, z.imag], axis=-1)
    np.testing.assert_allclose(oracle.rope_neox(x, pos, 1e6), ref, atol=1e-12)


# ---------------------------------------------------------------- attention
def _brute_attention(q, k, v, q_pos, k_pos):
    T, hq, d = q.shape
    hkv = k.shape[1]
    out = np.zeros_like(q)
    for t in range(T):
        for h in range(hq):
            g = h // (hq // hkv)
            js = [j for j in range(k.shape[0]) if k_pos[j] <= q_pos[t]]
            s = [sum(q[t, h, e] * k[j, g, e] for e in range(d)) / math.sqrt(d) for j in js]
            mx = max(s)
            w = [math.exp(si - mx) for si in s]
            tot = sum(w)
            for e in range(d):
                out[t, h, e] = sum(wi * v[j, g, e] for wi, j in zip(w, js)) / tot
    return out


def test_attention_brute_force_prefill_and_decode_rows():
    q = rng.normal(size=(5, 4, 8)); k = rng.normal(size=(5, 2, 8)); v = rng.normal(size=(5, 2, 8))
    pos = np.arange(5)
    np.testing.assert_allclose(oracle.causal_gqa_attention(q, k, v, pos, pos),
                               _brute_attention(q, k, v, pos, pos), rtol=1e-12, atol=1e-14)
    # a decode row at position 4 over keys 0..4
    np.testing.assert_allclose(oracle.causal_gqa_attention(q[4:], k, v, pos[4:], pos),
                               _brute_attention(q[4:], k, v, pos[4:], pos), rtol=1e-12, atol=1e-14)


def test_attention_matches_torch_sdpa():
    T, hq, hkv, d = 9, 4, 2, 16
    q = rng.normal(size=(T, hq, d)); k = rng.normal(size=(T, hkv, d)); v = rng.normal(size=(T, hkv, d))
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)[None]
    ref = Fn.scaled_dot_product_attention(tq, tk, tv, is_causal=True)[0].permute(1, 0, 2).numpy()
    pos = np.arange(T)
    np.testing.assert_allclose(oracle.causal_gqa_attention(q, k, v, pos, pos), ref, rtol=1e-12, atol=1e-13)


def test_softmax_rows_sum_to_one():
    q = rng.normal(size=(6, 4, 8)) * 5; k = rng.normal(size=(6, 2, 8)) * 5
    v = np.ones((6, 2, 8))
    out = oracle.causal_gqa_attention(q, k, v, np.arange(6), np.arange(6))
    np.testing.assert_allclose(out, 1.0, rtol=1e-14)


def test_attention_causality_and_single_key():
    q = rng.normal(size=(6, 4, 8)); k = rng.normal(size=(6, 2, 8)); v = rng.normal(size=(6, 2, 8))
    pos = np.arange(6)
    base = oracle.causal_gqa_attention(q, k, v, pos, pos)
    k2, v2 = k.copy(), v.copy()
    k2[4:] += 10.0; v2[4:] -= 3.0
    pert = oracle.causal_gqa_attention(q, k2, v2, pos, pos)
    assert np.array_equal(base[:4], pert[:4])
    assert not np.allclose(base[4:], pert[4:])
    # row 0 sees only key 0: output is v[0] of its kv head
    np.testing.assert_allclose(base[0, 0], v[0, 0], rtol=1e-15)
    np.testing.assert_allclose(base[0, 3], v[0, 1], rtol=1e-15)


def test_gqa_reduces_to_mha():
    q = rng.normal(size=(5, 4, 8)); k = rng.normal(size=(5, 2, 8)); v = rng.normal(size=(5, 2, 8))
    pos = np.arange(5)
    gqa = oracle.causal_gqa_attention(q, k, v, pos, pos)
    mha = oracle.causal_gqa_attention(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), pos, pos)
    np.testing.assert_allclose(gqa, mha, rtol=1e-15)


# ---------------------------------------------------------------- SwiGLU
def test_swiglu_closed_forms_and_order():
    F = 4
    gu = np.array([[0.0, 30.0, -30.0, 1.0, 2.0, 3.0, 4.0, 5.0]])
    y = oracle.swiglu(gu, F)[0]
    assert y[0] == 0.0                                # silu(0) = 0
    assert abs(y[1] - 30.0 * 3.0) < 1e-9              # silu(z) -> z for large z
    assert abs(y[2]) < 1e-9                           # silu(z) -> 0 for very negative z
    assert abs(y[3] - 1.0 / (1.0 + math.exp(-1.0)) * 5.0) < 1e-15
    x = rng.normal(size=(3, 2 * 16))
    ref = (Fn.silu(torch.from_numpy(x[:, :16])) * torch.from_numpy(x[:, 16:])).numpy()
    np.testing.assert_allclose(oracle.swiglu(x, 16), ref, rtol=1e-14)


# ---------------------------------------------------------------- splice / head / argmax
def test_inputs_embeds_replaces_rows():
    E = rng.normal(size=(50, 6))
    ids = np.array([3, 0, 0, 0, 7, 9])
    audio = rng.normal(size=(3, 6))
    x = oracle.inputs_embeds(E, ids, audio, 1)
    assert np.array_equal(x[0], E[3]) and np.array_equal(x[4], E[7]) and np.array_equal(x[5], E[9])
    assert np.array_equal(x[1:4], audio)
    x_end = oracle.inputs_embeds(E, ids, audio, 3)    # offset + n_audio == T
    assert np.array_equal(x_end[3:], audio) and np.array_equal(x_end[:3], E[ids[:3]])
    assert np.array_equal(oracle.inputs_embeds(E, ids, None, 0), E[ids])


def test_tied_head_matches_row_dots():
    E = rng.normal(size=(40, 12)); h = rng.normal(size=12)
    z = oracle.tied_lm_head(E, h)
    for r in (0, 17, 39):
        assert abs(z[r] - sum(E[r, i] * h[i] for i in range(12))) < 1e-12


def test_argmax_lowest_index_and_nan():
    assert oracle.greedy_argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.greedy_argmax([-1.0]) == 0
    with pytest.raises(FloatingPointError):
        oracle.greedy_argmax([0.0, float("nan")])


def test_fake_token_len_worked_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "fake_token_len.txt")) if l.strip() and not l.startswith("#")]
    for frames, n in rows:
        assert oracle.fake_token_len(int(frames)) == int(n)
    assert synth.WORKLOADS["funasr_nano_short"].n_audio == oracle.fake_token_len(183)


def test_step_metrics_hand_example():
    ref = np.array([1.0, -2.0, 0.0, 4.0]); cand = np.array([1.5, -2.0, 0.5, 4.0])
    m = oracle.step_metrics(cand, ref)
    assert m["max_abs"] == 0.5
    assert m["mean_abs"] == 0.25
    assert abs(m["rmse"] - math.sqrt(0.5 / 4)) < 1e-15
    assert abs(m["mean_rel"] - (0.5 + 0 + 0.5 / 1e-6 + 0) / 4) < 1e-6
    assert abs(m["cosine"] - (1.5 + 4 + 16) / (math.sqrt(21) * math.sqrt(2.25 + 4 + 0.25 + 16))) < 1e-15
    assert m["argmax_equal"] and m["top_gap_ref"] == 3.0
    ok, _ = oracle.parity_gate(cand, ref, 0.9995, 1e-2)
    assert not ok                                    # 0.5 > 1e-2 * 4
    ok, _ = oracle.parity_gate(ref + 0.01, ref, 0.9995, 1e-2)
    assert ok


# ---------------------------------------------------------------- whole decoder
@pytest.fixture(scope="module")
def tiny():
    w = synth.make_weights(synth.TINY, seed=0, gain_jitter=True)
    p = synth.make_prompt(synth.WORKLOADS["tiny"], seed=0)
    return w, p


def _np_weights(w):
    f = lambda t: t.to(torch.float64).numpy()
    return {"embed": f(w.embed), "final_norm": f(w.final_norm),
            "layers": [{k: f(v) for k, v in l.items()} for l in w.layers]}


def _torch_reference(shape, w, ids, audio, off, n_steps_tokens):
    """Independent float64 formulation: torch library rms_norm, SDPA (causal for
    the prompt, unmasked for one decode row over the full history) and silu;
    RoPE as complex multiplication; every step recomputes the whole sequence."""
    H, HQ, HKV, Dh, F = shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn
    t64 = lambda t: t.to(torch.float64)
    E = t64(w.embed)
    def forward(seq_ids):
        x = E[torch.as_tensor(seq_ids, dtype=torch.long)].clone()
        x[off:off + audio.shape[0]] = t64(audio)
        T = x.shape[0]
        pos = torch.arange(T, dtype=torch.float64)
        omega = torch.exp(-math.log(shape.rope_theta) * torch.arange(0, Dh, 2, dtype=torch.float64) / Dh)
        rot = torch.polar(torch.ones(T, Dh // 2, dtype=torch.float64), pos[:, None] * omega[None, :])
        def rope(a):   # [T, h, Dh]
            z = torch.complex(a[..., :Dh // 2], a[..., Dh // 2:]) * rot[:, None, :]
            return torch.cat([z.real, z.imag], dim=-1)
        for l in w.layers:
            xn = Fn.rms_norm(x, (H,), weight=t64(l["g_in"]), eps=shape.rms_eps)
            q, k, v = torch.split(xn @ t64(l["wqkv"]).T, [HQ * Dh, HKV * Dh, HKV * Dh], dim=-1)
            q = rope(Fn.rms_norm(q.reshape(T, HQ, Dh), (Dh,), weight=t64(l["g_q"]), eps=shape.rms_eps))
            k = rope(Fn.rms_norm(k.reshape(T, HKV, Dh), (Dh,), weight=t64(l["g_k"]), eps=shape.rms_eps))
            v = v.reshape(T, HKV, Dh)
            rep = HQ // HKV
            o = Fn.scaled_dot_product_attention(q.permute(1, 0, 2)[None],
                                                k.repeat_interleave(rep, 1).permute(1, 0, 2)[None],
                                                v.repeat_interleave(rep, 1).permute(1, 0, 2)[None],
                                                is_causal=True)[0].permute(1, 0, 2).reshape(T, HQ * Dh)
            x = x + o @ t64(l["wo"]).T
            xn = Fn.rms_norm(x, (H,), weight=t64(l["g_post"]), eps=shape.rms_eps)
            g, u = torch.split(xn @ t64(l["wgu"]).T, [F, F], dim=-1)
            x = x + (Fn.silu(g) * u) @ t64(l["wd"]).T
        h = Fn.rms_norm(x[-1], (H,), weight=t64(w.final_norm), eps=shape.rms_eps)
        return (E @ h).numpy()
    seq = list(ids)
    outs = [forward(seq)]
    for t in n_steps_tokens:
        seq.append(int(t))
        outs.append(forward(seq))
    return outs


def _oracle_run(o, ids, audio, off, toks):
    outs = [o.prefill(ids, audio, off)]
    for t in toks:
        outs.append(o.decode_step(t))
    return outs


def test_decoder_matches_independent_torch_formulation(tiny):
    w, p = tiny
    o = oracle.DecoderOracle(synth.TINY, _np_weights(w))
    toks = [5, 900, 17]
    ours = _oracle_run(o, p.ids.numpy(), p.audio.to(torch.float64).numpy(), p.audio_offset, toks)
    ref = _torch_reference(synth.TINY, w, p.ids.numpy(), p.audio, p.audio_offset, toks)
    for a, b in zip(ours, ref):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-10 * np.abs(b).max())


def test_splicing_embedding_rows_equals_text_prompt(tiny):
    w, p = tiny
    o = oracle.DecoderOracle(synth.TINY, _np_weights(w))
    ids = p.ids.numpy().copy()
    rows = np.arange(100, 108)
    ids_text = ids.copy(); ids_text[12:20] = rows
    a = o.prefill(ids, o.embed[rows], 12)
    b = o.prefill(ids_text, None, 0)
    assert np.array_equal(a, b)


def test_incremental_decode_equals_full_recompute(tiny):
    w, p = tiny
    o = oracle.DecoderOracle(synth.TINY, _np_weights(w))
    ids = p.ids.numpy(); audio = p.audio.to(torch.float64).numpy()
    z = o.prefill(ids, audio, p.audio_offset)
    seq = list(ids)
    for _ in range(6):
        t = oracle.greedy_argmax(z)
        z = o.decode_step(t)
        seq.append(t)
        full = o.full_recompute(seq, audio, p.audio_offset)
        np.testing.assert_allclose(z, full, rtol=0, atol=1e-10 * np.abs(full).max())
    assert o.position == len(seq) and o.history == seq


def test_clone_then_decode_equals_decode(tiny):
    w, p = tiny
    o = oracle.DecoderOracle(synth.TINY, _np_weights(w))
    o.prefill(p.ids.numpy(), p.audio.to(torch.float64).numpy(), p.audio_offset)
    c = o.clone()
    a = [o.decode_step(t) for t in (1, 2, 3)]
    b = [c.decode_step(t) for t in (1, 2, 3)]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    with pytest.raises(RuntimeError):
        oracle.DecoderOracle(synth.TINY, _np_weights(w)).decode_step(1)


# ---------------------------------------------------------------- planted mistakes
_rope, _attn, _swiglu, _rms = od.rope_neox, od.causal_gqa_attention, od.swiglu, od.rms_norm


def _plant_rope_sign(x, positions, theta):
    return _rope(x, -np.asarray(positions), theta)

def _plant_rope_interleaved(x, positions, theta):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    inv = np.argsort(perm)
    return _rope(x[..., perm], positions, theta)[..., inv]

def _plant_gqa_modulo(q, k, v, q_pos, k_pos):
    hq, hkv = q.shape[1], k.shape[1]
    idx = np.arange(hq) % hkv                      # wrong grouping (tile instead of repeat)
    return _attn(q, np.asarray(k)[:, idx], np.asarray(v)[:, idx], q_pos, k_pos)

def _plant_no_causal(q, k, v, q_pos, k_pos):
    return _attn(q, k, v, np.full(len(q_pos), 10 ** 9), k_pos)

def _plant_swap_gate_up(gu, ffn):
    gu = np.asarray(gu, np.float64)
    return _swiglu(np.concatenate([gu[..., ffn:], gu[..., :ffn]], axis=-1), ffn)

def _plant_rms_no_eps(x, gain, eps):
    return _rms(x, gain, 0.0) * (1.0 + 1e-3)


@pytest.mark.parametrize("name,target,fake", [
    ("rope_sign", "rope_neox", _plant_rope_sign),
    ("rope_interleaved", "rope_neox", _plant_rope_interleaved),
    ("gqa_modulo", "causal_gqa_attention", _plant_gqa_modulo),
    ("no_causal_mask", "causal_gqa_attention", _plant_no_causal),
    ("swapped_gate_up", "swiglu", _plant_swap_gate_up),
    ("rms_scale", "rms_norm", _plant_rms_no_eps),
])
def test_planted_mistake_is_caught(tiny, monkeypatch, name, target, fake):
    w, p = tiny
    monkeypatch.setattr(od, target, fake)
    o = oracle.DecoderOracle(synth.TINY, _np_weights(w))
    toks = [5, 900]
    ours = _oracle_run(o, p.ids.numpy(), p.audio.to(torch.float64).numpy(), p.audio_offset, toks)
    ref = _torch_reference(synth.TINY, w, p.ids.numpy(), p.audio, p.audio_offset, toks)
    worst = max(float(np.abs(a - b).max() / np.abs(b).max()) for a, b in zip(ours, ref))
    assert worst > 1e-6, f"planted mistake {name} not detected"
