"""GPU token choice (qdec_op_sample, qdec_set_sampling) against the float64 sampling
oracle on the same fp32 logits ("Qwen3ASR ncnn多平台移植" §1 and §6: greedy, temperature,
top-k, top-p and repetition penalty).  The choice is an integer decided by floating point:
the GPU's pick must equal the oracle's, except where the draw u falls within 1e-5 of a
boundary of the oracle's cumulative distribution, where either neighbour is correct."""
import numpy as np
import pytest
import torch

from oracle import sampling as S
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Decoder, QdecError

import _harness as H

pytestmark = pytest.mark.gpu


def _valid(z, hist, t, k, p, r, seed, pos, got):
    exp = S.sample_token(z, hist, t, k, p, r, seed, pos)
    if got == exp:
        return True
    if t == 0.0:
        return False
    zz = S.repetition_penalty(z, hist, r) / t
    keep = S.top_p_mask(zz, S.top_k_mask(zz, k), p)
    if not keep[got]:
        return False
    w = np.where(keep, np.exp(zz - zz[keep].max()), 0.0)
    c = np.cumsum(w) / w.sum()
    u = S.counter_uniform(seed, pos)
    return c[got] - w[got] / w.sum() - 1e-5 <= u <= c[got] + 1e-5


CASES = [(0.0, 0, 1.0, 1.0), (1.0, 0, 1.0, 1.0), (0.7, 40, 1.0, 1.0), (1.0, 0, 0.9, 1.0), (0.8, 50, 0.95, 1.3),
         (1.5, 1, 1.0, 1.0), (1.0, 0, 1e-6, 1.0), (0.0, 0, 1.0, 2.0), (1.2, 200, 0.5, 1.1)]


@pytest.mark.parametrize("V", [1000, 151936])
@pytest.mark.parametrize("t,k,p,r", CASES)
def test_sample_op_matches_oracle(V, t, k, p, r):
    rng = np.random.default_rng(V + int(1000 * t) + k)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for trial in range(6):
        z = (rng.normal(size=V) * rng.choice([0.6, 3.0])).astype(np.float32)
        hist = rng.integers(0, V, size=int(rng.integers(1, 40))).astype(np.int32)
        seed, pos = int(rng.integers(0, 2**63)), int(rng.integers(0, 4096))
        _lib.sample(torch.from_numpy(z).cuda(), V, torch.from_numpy(hist).cuda(), t, k, p, r, seed, pos, tok)
        torch.cuda.synchronize()
        got = int(tok.item())
        assert _valid(z.astype(np.float64), hist, t, k, p, r, seed, pos, got), (trial, got)


@pytest.mark.parametrize("V", [1000, 151936])
def test_sample_op_top_k_keeps_ties(V):
    """Logits quantised to a few levels make the k-th largest value a tie group: every member
    of it stays in the top-k set, so the draws cover ids past the first k and each pick is the
    oracle's."""
    rng = np.random.default_rng(V)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    z = np.round(rng.normal(size=V) * 2.0).astype(np.float32)          # many equal values
    k = int((z >= np.sort(z)[::-1][20]).sum()) - 3                     # k ends inside a tie group
    keep = S.top_k_mask(z.astype(np.float64), k)
    assert keep.sum() > k                                              # the oracle keeps the whole group
    zt = torch.from_numpy(z).cuda()
    seen = set()
    for pos in range(64):
        _lib.sample(zt, V, None, 1.0, k, 1.0, 1.0, 5, pos, tok)
        torch.cuda.synchronize()
        got = int(tok.item())
        assert keep[got], (pos, got)
        assert _valid(z.astype(np.float64), np.zeros(0, np.int32), 1.0, k, 1.0, 1.0, 5, pos, got), (pos, got)
        seen.add(got)
    assert len(seen) > 1


def test_sample_op_full_vocab_top_p_with_penalty():
    """Top-p over the full 151,936-entry vocabulary with a long history under the repetition
    penalty: the penalised ids' logits move before the nucleus is cut."""
    V = 151936
    rng = np.random.default_rng(3)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for trial in range(8):
        z = (rng.normal(size=V) * 4.0).astype(np.float32)
        top = np.argsort(-z)[:64]
        hist = np.concatenate([top[:32], rng.integers(0, V, size=400)]).astype(np.int32)
        seed, pos = int(rng.integers(0, 2**63)), int(rng.integers(0, 8192))
        for p in (0.5, 0.9, 0.99):
            _lib.sample(torch.from_numpy(z).cuda(), V, torch.from_numpy(hist).cuda(), 0.8, 0, p, 1.5, seed, pos, tok)
            torch.cuda.synchronize()
            got = int(tok.item())
            assert _valid(z.astype(np.float64), hist, 0.8, 0, p, 1.5, seed, pos, got), (trial, p, got)


def test_sample_op_is_deterministic_and_draws_per_position():
    rng = np.random.default_rng(1)
    z = torch.from_numpy((rng.normal(size=5000) * 0.5).astype(np.float32)).cuda()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    picks = []
    for pos in range(40):
        a = []
        for _ in range(2):
            _lib.sample(z, 5000, None, 1.0, 0, 1.0, 1.0, 99, pos, tok)
            a.append(int(tok.item()))
        assert a[0] == a[1]
        picks.append(a[0])
    assert len(set(picks)) > 20   # different positions draw different tokens from a flat distribution


def test_sample_op_rejects_bad_parameters():
    z = torch.zeros(10, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t, k, p, r in [(-1.0, 0, 1.0, 1.0), (1.0, -1, 1.0, 1.0), (1.0, 0, 0.0, 1.0), (1.0, 0, 1.5, 1.0),
                       (1.0, 0, 1.0, 0.0)]:
        with pytest.raises(QdecError):
            _lib.sample(z, 10, None, t, k, p, r, 0, 0, tok)


@pytest.fixture(scope="module")
def tiny():
    w = synth.make_weights(synth.TINY, seed=0)
    return w, w.to("cuda")


def _prompt():
    wl = synth.Workload("t", synth.TINY, 12, 8, 12, 0)
    return synth.make_prompt(wl, 0)


@pytest.mark.parametrize("kernel", [_lib.DECODE_PERSISTENT, _lib.DECODE_GRAPH], ids=["persistent", "graph"])
def test_decoder_sampling_trajectory(tiny, kernel):
    """Prefill and steps with token = -1 feed the sampled token back on the device; each
    choice is the oracle's choice on the returned logits and the recorded history, drawn at
    the logits row's position."""
    w, wd = tiny
    p = _prompt()
    T = p.ids.numel()
    t, k, pp, r, seed = 0.9, 50, 0.95, 1.2, 12345
    dec = Decoder(synth.TINY, wd, max_seq=T + 20)
    dec.decode_kernel = kernel
    dec.set_sampling(t, k, pp, r, seed)
    lg = torch.empty(synth.TINY.vocab, device="cuda")
    a = dec.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=lg)
    hist = dec.read_history(T)
    assert _valid(lg.cpu().double().numpy(), hist, t, k, pp, r, seed, T - 1, a)
    fed = [a]
    for step in range(16):
        pos = T + step
        a = dec.decode_step(-1, logits=lg)
        hist = dec.read_history(pos + 1)
        assert hist[pos] == fed[-1]   # the previous choice was fed back
        assert _valid(lg.cpu().double().numpy(), hist, t, k, pp, r, seed, pos, a), step
        fed.append(a)


def test_greedy_setting_matches_default(tiny):
    w, wd = tiny
    p = _prompt()
    a = Decoder(synth.TINY, wd, max_seq=40)
    b = Decoder(synth.TINY, wd, max_seq=40)
    b.set_sampling(0.0, 0, 1.0, 1.0, 7)
    ta = [a.prefill(p.ids, p.audio.cuda(), p.audio_offset)]
    tb = [b.prefill(p.ids, p.audio.cuda(), p.audio_offset)]
    for _ in range(5):
        ta.append(a.decode_step(-1))
        tb.append(b.decode_step(-1))
    assert ta == tb


def test_batch_step_rejects_sampling_contexts(tiny):
    w, wd = tiny
    p = _prompt()
    a = Decoder(synth.TINY, wd, max_seq=40)
    a.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    b = a.clone()
    b.set_sampling(1.0, 0, 1.0, 1.0, 3)
    with pytest.raises(QdecError):
        Decoder.decode_step_batch([a, b], [1, 2])
    with pytest.raises(QdecError):
        a.set_sampling(-0.5, 0, 1.0, 1.0, 0)
