"""GPU parity on the tiny Qwen3-style decoder (hidden 128, 2 layers, 4/2 heads,
head_dim 32, ffn 384, vocab 1024): every call goes through the C ABI and is
compared with the float64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Decoder, QdecError, DECODE_PERSISTENT, DECODE_GRAPH

import _harness as H

pytestmark = pytest.mark.gpu
SH = synth.TINY


@pytest.fixture(scope="module")
def model():
    w = synth.make_weights(SH, seed=0)
    return w, w.to("cuda"), H.make_oracle(w)


@pytest.fixture(scope="module")
def model_jitter():
    w = synth.make_weights(SH, seed=5, gain_jitter=True)
    return w, w.to("cuda"), H.make_oracle(w)


def _prompt(n_prefix, n_audio, n_suffix, seed=0):
    wl = synth.Workload("t", SH, n_prefix, n_audio, n_suffix, 0)
    return synth.make_prompt(wl, seed)


LAYOUTS = [(12, 8, 12, 16),     # the tiny workload: 32 positions, 16 steps
           (12, 50, 15, 8),     # 77 positions: two 64-row tiles + ragged tail
           (0, 20, 5, 4),       # audio at offset 0
           (10, 6, 0, 4),       # audio ends at the last position
           (40, 0, 0, 4),       # text only
           (1, 0, 0, 3),        # a single-token prompt
           (3, 130, 2, 2),      # 135 positions
           (3, 590, 7, 4)]      # 600 positions: decode attention split over several key chunks


@pytest.mark.parametrize("kernel", [DECODE_PERSISTENT, DECODE_GRAPH], ids=["persistent", "graph"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_teacher_forced_logits(model, layout, kernel):
    w, wd, orc = model
    n_prefix, n_audio, n_suffix, steps = layout
    p = _prompt(n_prefix, n_audio, n_suffix)
    dec = Decoder(SH, wd, max_seq=p.ids.numel() + steps)
    dec.decode_kernel = kernel
    assert dec.decode_kernel == kernel
    res = H.teacher_forced(dec, orc, p, steps)
    H.assert_step_parity(res, f"tiny {layout}")
    assert dec.position == p.ids.numel() + steps


def test_persistent_kernel_is_the_default(model):
    w, wd, orc = model
    dec = Decoder(SH, wd, max_seq=40)
    assert dec.decode_kernel == DECODE_PERSISTENT
    assert dec.clone().decode_kernel == DECODE_PERSISTENT
    dec.decode_kernel = DECODE_GRAPH
    assert dec.clone().decode_kernel == DECODE_GRAPH
    with pytest.raises(QdecError):
        dec.decode_kernel = 7


def test_gain_jitter(model_jitter):
    w, wd, orc = model_jitter
    p = _prompt(12, 8, 12)
    dec = Decoder(SH, wd, max_seq=48)
    H.assert_step_parity(H.teacher_forced(dec, orc, p, 8), "tiny gains")


def test_kv_slots_match_oracle_positions(model):
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    steps = 5
    dec = Decoder(SH, wd, max_seq=64)
    H.teacher_forced(dec, orc, p, steps)
    L = p.ids.numel() + steps
    for l in range(SH.n_layers):
        for kind, ref in ((0, orc.k_cache[l]), (1, orc.v_cache[l])):
            got = dec.read_kv(l, kind, 0, 64)                       # [HKV, 64, D] bf16 bits
            g = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            assert not g[:, L:].any(), "slots beyond the written positions must stay untouched"
            r = np.transpose(ref, (1, 0, 2))                        # [HKV, L, D]
            gl = g[:, :L]
            assert np.abs(gl - r).max() <= 2e-2 * np.abs(r).max()
            # slot index == absolute position: each slot's own position attains the minimum
            # distance (V rows of repeated tokens can coincide, so ties are allowed)
            for h in range(SH.n_kv_heads):
                d = ((gl[h][:, None, :] - r[h][None, :, :]) ** 2).sum(-1)
                own = d[np.arange(L), np.arange(L)]
                assert np.all(own <= d.min(axis=1) + 1e-12)
                if kind == 0:   # RoPE makes every position's key distinct: strict
                    assert np.array_equal(d.argmin(axis=1), np.arange(L))


def test_history_and_device_feedback(model):
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    a = Decoder(SH, wd, max_seq=48)
    b = Decoder(SH, wd, max_seq=48)
    la = torch.empty(SH.vocab, device="cuda")
    lb = torch.empty(SH.vocab, device="cuda")
    ta = a.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    tb = b.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    assert ta == tb
    for _ in range(10):
        a.decode_step(-1, want_argmax=False)          # greedy feedback stays on the device
        tb = b.decode_step(tb, logits=lb)             # host round trip
    a.decode_step(-1, logits=la, want_argmax=False)
    b.decode_step(tb, logits=lb)
    ha, hb = a.read_history(), b.read_history()
    assert np.array_equal(ha, hb)
    assert np.array_equal(ha[:12], p.ids.numpy()[:12])
    assert torch.equal(la, lb)


def test_repeat_runs_are_bitwise_identical(model):
    w, wd, orc = model
    p = _prompt(12, 50, 15)
    outs = []
    for _ in range(2):
        dec = Decoder(SH, wd, max_seq=80)
        lg = torch.empty(SH.vocab, device="cuda")
        dec.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=lg)
        seq = [lg.clone()]
        for t in (3, 4, 5):
            dec.decode_step(t, logits=lg)
            seq.append(lg.clone())
        outs.append(torch.stack(seq))
    assert torch.equal(outs[0], outs[1])


def test_host_and_device_buffers_agree(model):
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    d1 = Decoder(SH, wd, max_seq=40)
    d2 = Decoder(SH, wd, max_seq=40)
    l1 = torch.empty(SH.vocab, device="cuda")
    l2 = torch.empty(SH.vocab).pin_memory()
    l3 = torch.empty(SH.vocab)                      # pageable host memory
    a1 = d1.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=l1)
    a2 = d2.prefill(p.ids, p.audio, p.audio_offset, logits=l2)     # host audio rows
    assert a1 == a2 and torch.equal(l1.cpu(), l2)
    d1.decode_step(7, logits=l1)
    d2.decode_step(7, logits=l3)
    assert torch.equal(l1.cpu(), l3)


def test_clone_branches(model):
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    src = Decoder(SH, wd, max_seq=48)
    src.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    o_src = orc.clone(); o_src.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    c1 = src.clone()
    assert c1.position == src.position
    lg_a = torch.empty(SH.vocab, device="cuda"); lg_b = torch.empty(SH.vocab, device="cuda")
    # identical inputs: clone and source stay bitwise equal
    src.decode_step(11, logits=lg_a); c1.decode_step(11, logits=lg_b)
    assert torch.equal(lg_a, lg_b)
    # divergent branches each match an oracle branch
    o_a = o_src.clone(); o_b = o_src.clone()
    za = o_a.decode_step(11); zb = o_b.decode_step(11)
    for ta, tb in ((20, 900), (21, 901), (22, 902)):
        src.decode_step(ta, logits=lg_a); c1.decode_step(tb, logits=lg_b)
        za = o_a.decode_step(ta); zb = o_b.decode_step(tb)
        for g, r in ((lg_a, za), (lg_b, zb)):
            ok, m = oracle.parity_gate(g.cpu().numpy(), r, H.COS_MIN, H.REL_BOUND)
            assert ok, m
    assert src.read_history()[-3:].tolist() == [20, 21, 22]
    assert c1.read_history()[-3:].tolist() == [900, 901, 902]


def test_batch_step_matches_single_streams(model):
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    src = Decoder(SH, wd, max_seq=48)
    src.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    o_src = orc.clone(); o_src.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    n = 5
    branches = [src.clone() for _ in range(n)]
    singles = [src.clone() for _ in range(n)]
    obr = [o_src.clone() for _ in range(n)]
    toks = synth.make_tokens(SH.vocab, n, seed=3).numpy()
    lb = torch.empty(n, SH.vocab, device="cuda")
    ls = torch.empty(SH.vocab, device="cuda")
    for step in range(4):
        am = Decoder.decode_step_batch(branches, toks, logits=lb)
        for i in range(n):
            a1 = singles[i].decode_step(int(toks[i]), logits=ls)
            z = obr[i].decode_step(int(toks[i]))
            ok, m = oracle.parity_gate(lb[i].cpu().numpy(), z, H.COS_MIN, H.REL_BOUND)
            assert ok, (step, i, m)
            assert am[i] == int(torch.argmax(lb[i]))
            # the batch runs its projections on the tensor cores with bf16 activations, a
            # single step keeps them fp32: they agree to bf16 rounding
            np.testing.assert_allclose(lb[i].cpu().numpy(), ls.cpu().numpy(), rtol=0,
                                       atol=1e-2 * float(ls.abs().max()))
        toks = am                                    # greedy continuation per stream
    assert all(b.position == p.ids.numel() + 4 for b in branches)


def test_batch_graph_follows_composition_and_options(model):
    """The lockstep step is replayed from a graph after its first step; a new batch
    composition or a GEMM-implementation change must rebuild it, with the argmax fed back
    on the device (token -1) throughout."""
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    src = Decoder(SH, wd, max_seq=48)
    src.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    A = [src.clone() for _ in range(3)]
    S = [src.clone() for _ in range(3)]
    first = synth.make_tokens(SH.vocab, 3, seed=5).numpy()
    lb = torch.empty(3, SH.vocab, device="cuda")
    ls = torch.empty(SH.vocab, device="cuda")

    def check(batch, singles, toks, single_toks, k):
        # the batch feeds its own argmax back on the device (token -1); the single streams get
        # the batch's previous picks explicitly, so near ties cannot make the two diverge
        am = Decoder.decode_step_batch(batch, toks, logits=lb[:len(batch)])
        for i, sd in enumerate(singles):
            sd.decode_step(int(single_toks[i]), logits=ls)
            np.testing.assert_allclose(lb[i].cpu().numpy(), ls.cpu().numpy(), rtol=0,
                                       atol=1e-2 * float(ls.abs().max()), err_msg=f"step {k} stream {i}")
            assert am[i] == int(torch.argmax(lb[i]))
        return am

    am = check(A, S, first, first, 0)
    for k in range(1, 4):                                # eager, captured, replayed
        am = check(A, S, np.full(3, -1, dtype=np.int32), am, k)
    am2 = am[[0, 2]]
    for k in range(4, 7):                                # new composition
        am2 = check([A[0], A[2]], [S[0], S[2]], np.full(2, -1, dtype=np.int32), am2, k)
    A[0].set_option(_lib.OPT_PREFILL_IMPL, _lib.PREFILL_SIMT)
    for k in range(7, 9):                                # CUDA-core GEMMs
        am2 = check([A[0], A[2]], [S[0], S[2]], np.full(2, -1, dtype=np.int32), am2, k)
    assert A[0].position == A[2].position == p.ids.numel() + 9 and A[1].position == p.ids.numel() + 4
    assert np.array_equal(A[0].read_history(), S[0].read_history())


def test_errors_leave_context_unchanged(model):
    w, wd, orc = model
    p = _prompt(12, 8, 12)
    dec = Decoder(SH, wd, max_seq=33)
    with pytest.raises(QdecError) as e:
        dec.decode_step(1)
    assert e.value.status == -3                      # decode before prefill
    bad = p.ids.clone(); bad[3] = SH.vocab
    with pytest.raises(QdecError) as e:
        dec.prefill(bad, p.audio.cuda(), p.audio_offset)
    assert e.value.status == -1
    with pytest.raises(QdecError) as e:
        dec.prefill(p.ids, p.audio.cuda(), 30)       # audio rows past the prompt end
    assert e.value.status == -1
    long_ids = torch.zeros(34, dtype=torch.int32)
    with pytest.raises(QdecError) as e:
        dec.prefill(long_ids)
    assert e.value.status == -2
    dec.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    assert dec.position == 32
    with pytest.raises(QdecError) as e:
        dec.decode_step(-2)
    assert e.value.status == -1
    with pytest.raises(QdecError) as e:
        dec.decode_step(SH.vocab)
    assert e.value.status == -1
    assert dec.position == 32
    dec.decode_step(5)
    with pytest.raises(QdecError) as e:
        dec.decode_step(6)                           # slot 33 >= max_seq
    assert e.value.status == -2
    assert dec.position == 33


@pytest.mark.parametrize("keys", [8, 24, 4096])
def test_attention_unit_size_option(model, keys):
    """QDEC_OPT_ATTN_UNIT_KEYS only changes how the persistent step splits the KV history
    into attention units (and so the summation order): logits agree with the default split
    to fp32 rounding, teacher-forced parity against the oracle holds, and clones inherit it."""
    w, wd, orc = model
    p = _prompt(12, 50, 15)
    a = Decoder(SH, wd, max_seq=p.ids.numel() + 6)
    b = Decoder(SH, wd, max_seq=p.ids.numel() + 6)
    b.set_option(_lib.OPT_ATTN_UNIT_KEYS, keys)
    assert b.get_option(_lib.OPT_ATTN_UNIT_KEYS) == keys
    la = torch.empty(SH.vocab, device="cuda"); lb = torch.empty(SH.vocab, device="cuda")
    a.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    b.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    c = b.clone()
    assert c.get_option(_lib.OPT_ATTN_UNIT_KEYS) == keys
    for t in (5, 9, 13, 2):
        ta = a.decode_step(t, logits=la)
        tb = b.decode_step(t, logits=lb)
        ga, gb = la.cpu().double().numpy(), lb.cpu().double().numpy()
        assert np.abs(ga - gb).max() <= 1e-4 * np.abs(ga).max()
        assert tb == int(np.argmax(gb))
    d = Decoder(SH, wd, max_seq=p.ids.numel() + 6)
    d.set_option(_lib.OPT_ATTN_UNIT_KEYS, keys)
    H.assert_step_parity(H.teacher_forced(d, orc, p, 5), f"tiny unit keys {keys}")


def test_attention_unit_size_option_rejects_bad_values(model):
    w, wd, orc = model
    d = Decoder(SH, wd, max_seq=40)
    for v in (-8, 4, 12, 4104):
        with pytest.raises(QdecError):
            d.set_option(_lib.OPT_ATTN_UNIT_KEYS, v)
    assert d.get_option(_lib.OPT_ATTN_UNIT_KEYS) == 0


def test_repeated_prefill_replays_identically(model):
    """The second prefill of a prompt length is captured as a CUDA graph and later ones
    replay it: logits, argmax and the decode steps that follow are bitwise those of the
    first (eager) prefill, also when other lengths are prefilled in between."""
    w, wd, orc = model
    p = _prompt(12, 50, 15)
    q = _prompt(3, 20, 4, seed=1)
    dec = Decoder(SH, wd, max_seq=p.ids.numel() + 4)
    lg = torch.empty(SH.vocab, device="cuda")
    runs = []
    for i in range(4):
        if i == 2:
            dec.prefill(q.ids, q.audio.cuda(), q.audio_offset)   # another length in between
        a = dec.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=lg)
        seq = [lg.clone()]
        toks = [a]
        for t in (3, -1, -1):
            toks.append(dec.decode_step(t, logits=lg))
            seq.append(lg.clone())
        runs.append((toks, torch.stack(seq)))
        assert dec.position == p.ids.numel() + 3
    for toks, seq in runs[1:]:
        assert toks == runs[0][0]
        assert torch.equal(seq, runs[0][1])
    H.assert_step_parity(H.teacher_forced(dec, orc, p, 3), "tiny prefill replay")
