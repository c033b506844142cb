"""Full-size parity (Qwen3-0.6B shape: hidden 1024, 28 layers, GQA 16/8, head_dim
128, ffn 3072, vocab 151936) on the workloads' own prompt layouts, teacher-forced
against the float64 oracle ("Qwen3ASR ncnn多平台移植" §7.1-§7.2)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Decoder, DECODE_PERSISTENT, DECODE_GRAPH

import _harness as H

pytestmark = pytest.mark.gpu
SH = synth.QWEN3_06B


@pytest.fixture(scope="module")
def full():
    w = synth.make_weights(SH, seed=0)
    return w, w.to("cuda"), H.make_oracle(w)


def _report(name, res):
    out = os.environ.get("QDEC_PARITY_REPORT_DIR")
    ms = [oracle.step_metrics(g, r) for g, r, _ in res]
    summary = {"workload": name, "steps": len(ms),
               "min_cosine": min(m["cosine"] for m in ms),
               "max_abs_over_max_ref": max(m["max_abs"] / m["max_abs_ref"] for m in ms),
               "mean_abs": float(np.mean([m["mean_abs"] for m in ms])),
               "rmse": float(np.mean([m["rmse"] for m in ms])),
               "max_mean_rel": max(m["mean_rel"] for m in ms),
               "argmax_agreement": float(np.mean([m["argmax_equal"] for m in ms]))}
    print(json.dumps(summary))
    if out:
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, f"parity_{name}.json"), "w") as f:
            json.dump({"summary": summary, "per_step": ms}, f, indent=1)
    return summary


@pytest.mark.parametrize("name", ["funasr_nano_short", "qwen3_asr_30s"])
def test_teacher_forced_workload(full, name):
    w, wd, orc = full
    wl = synth.WORKLOADS[name]
    p = synth.make_prompt(wl, seed=0)
    dec = Decoder(SH, wd, max_seq=wl.max_seq)
    res = H.teacher_forced(dec, orc.clone(), p, wl.n_decode)
    H.assert_step_parity(res, name)
    _report(name, res)
    hist = dec.read_history()
    assert hist.size == wl.max_seq
    kv_prompt = p.ids.numpy().copy()
    mask = np.ones(kv_prompt.size, bool); mask[wl.audio_offset:wl.audio_offset + wl.n_audio] = False
    assert np.array_equal(hist[:wl.n_prompt][mask], kv_prompt[mask])


@pytest.mark.parametrize("name,tile", [("funasr_nano_short", 0), ("qwen3_asr_30s", 0), ("qwen3_asr_30s", 256),
                                       ("qwen3_asr_30s", 256256), ("qwen3_asr_30s", 128)])
def test_fused_qkv_epilogue_matches_separate_kernels(full, name, tile):
    """The tcgen05 prefill writes K and V from the QKV GEMM's epilogue (per-head norm + RoPE
    fused); the CUDA-core prefill runs the GEMM and the norm/RoPE/append kernel separately.
    Both caches and the prefill logits must agree to bf16 rounding.  tile=256 forces the
    128 x 256 GEMM tiles (two heads per tile) that long prompts use, 256256 the 256 x 256
    tiles on a CTA pair of the longest prompts."""
    w, wd, orc = full
    wl = synth.WORKLOADS[name]
    p = synth.make_prompt(wl, seed=0)
    decs, logits = [], []
    for impl in (_lib.PREFILL_TCGEN05, _lib.PREFILL_SIMT):
        d = Decoder(SH, wd, max_seq=wl.n_prompt + 1)
        d.set_option(_lib.OPT_PREFILL_IMPL, impl)
        lg = torch.empty(SH.vocab, device="cuda")
        prev = _lib.gemm_tile_width(tile % 1000)
        prev_rows = _lib.gemm_tile_rows(tile // 1000)
        try:
            d.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=lg)
            d.sync()
        finally:
            _lib.gemm_tile_width(prev)
            _lib.gemm_tile_rows(prev_rows)
        decs.append(d)
        logits.append(lg.cpu().numpy())
    for layer in (0, 13, SH.n_layers - 1):
        for kind in (0, 1):
            a = decs[0].read_kv(layer, kind, 0, wl.n_prompt).view(np.uint16).astype(np.uint32) << 16
            b = decs[1].read_kv(layer, kind, 0, wl.n_prompt).view(np.uint16).astype(np.uint32) << 16
            fa, fb = a.view(np.float32), b.view(np.float32)
            np.testing.assert_allclose(fa, fb, rtol=0, atol=1e-2 * float(np.abs(fb).max()),
                                       err_msg=f"layer {layer} kind {kind}")
            # the epilogue's bulk stores end at the prompt: the slot after it is still zero
            assert not decs[0].read_kv(layer, kind, wl.n_prompt, 1).any(), f"layer {layer} kind {kind}"
    np.testing.assert_allclose(logits[0], logits[1], rtol=0, atol=1e-2 * float(np.abs(logits[1]).max()))


def test_persistent_and_graph_decode_agree(full):
    """The persistent single-kernel step and the per-op graph step compute the same
    function; with different summation orders they agree to fp32 rounding."""
    w, wd, orc = full
    wl = synth.WORKLOADS["qwen3_asr_30s"]
    p = synth.make_prompt(wl, seed=1)
    a = Decoder(SH, wd, max_seq=wl.max_seq)
    b = Decoder(SH, wd, max_seq=wl.max_seq)
    assert a.decode_kernel == DECODE_PERSISTENT
    b.decode_kernel = DECODE_GRAPH
    la = torch.empty(SH.vocab, device="cuda"); lb = torch.empty(SH.vocab, device="cuda")
    ta = a.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    b.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    for t in synth.make_tokens(SH.vocab, 12, seed=7).tolist():
        a.decode_step(t, logits=la)
        b.decode_step(t, logits=lb)
        ga, gb = la.cpu().double().numpy(), lb.cpu().double().numpy()
        assert np.abs(ga - gb).max() <= 1e-3 * np.abs(gb).max()
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for l in (0, 13, 27):
        for kind in (0, 1):
            ka = f(a.read_kv(l, kind, 0, wl.n_prompt + 12))
            kb = f(b.read_kv(l, kind, 0, wl.n_prompt + 12))
            assert np.array_equal(ka[:, :wl.n_prompt], kb[:, :wl.n_prompt])     # same prefill kernels
            assert np.abs(ka - kb).max() <= 2e-2 * np.abs(kb).max()


def test_mid_length_prefill(full):
    """A 1100-position prompt (30 ids, 1040 audio rows, 30 ids): every projection has enough
    tiles to run unsplit on 128 x 256 tiles, and attention spans nine 128-key tiles.  Logits
    of the prefill and two decode steps against the oracle; KV slots of the first, middle and
    last layer against the CUDA-core prefill: each path is within 1e-2 of max|ref| of the exact
    slots (one bf16 rounding per operand over the layers), so the two agree to the sum, 2e-2."""
    w, wd, orc = full
    wl = synth.Workload("mid", SH, 30, 1040, 30, 2)
    p = synth.make_prompt(wl, seed=3)
    dec = Decoder(SH, wd, max_seq=wl.max_seq)
    res = H.teacher_forced(dec, orc.clone(), p, 2)
    H.assert_step_parity(res, "1100 positions")
    _report("prefill_1100", res)
    ref = Decoder(SH, wd, max_seq=wl.n_prompt)
    ref.set_option(_lib.OPT_PREFILL_IMPL, _lib.PREFILL_SIMT)
    ref.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32)
    for layer in (0, 13, SH.n_layers - 1):
        for kind in (0, 1):
            a = f(dec.read_kv(layer, kind, 0, wl.n_prompt))
            b = f(ref.read_kv(layer, kind, 0, wl.n_prompt))
            np.testing.assert_allclose(a, b, rtol=0, atol=2e-2 * float(np.abs(b).max()), err_msg=f"{layer} {kind}")


@pytest.mark.parametrize("name", ["funasr_nano_short", "qwen3_asr_30s", "long_context"])
def test_programmatic_launch_is_bit_identical(full, name):
    """The prefill chain launched with programmatic dependent launch (each kernel starts its
    prologue and first weight loads while the previous one finishes, then waits for it) and
    launched plainly must give the same bits: logits of the eager run, the captured run and
    the graph replay, and every layer's K and V slots.  64 positions take the split-K paths,
    415 a mix, 4096 the unsplit 128 x 256 tiles."""
    w, wd, orc = full
    wl = synth.WORKLOADS[name]
    p = synth.make_prompt(wl, seed=0)
    runs = []
    for on in (1, 0):
        prev = _lib.programmatic_launch(on)
        try:
            d = Decoder(SH, wd, max_seq=wl.n_prompt + 1)
            lg = torch.empty(SH.vocab, device="cuda")
            logits = []
            for _ in range(3):   # eager, captured into a graph, replayed
                d.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=lg)
                d.sync()
                logits.append(lg.cpu().numpy().copy())
            _lib.device_error()
            kv = [d.read_kv(l, k, 0, wl.n_prompt) for l in range(SH.n_layers) for k in (0, 1)]
            d.close()
        finally:
            _lib.programmatic_launch(prev)
        runs.append((logits, kv))
    (la, ka), (lb, kb) = runs
    for i in range(3):
        assert np.array_equal(la[i].view(np.uint32), lb[i].view(np.uint32)), f"logits of run {i}"
        assert np.array_equal(la[i].view(np.uint32), la[0].view(np.uint32)), f"run {i} against the eager run"
    for i, (a, b) in enumerate(zip(ka, kb)):
        assert np.array_equal(a, b), f"layer {i // 2} kind {i % 2}"


@pytest.mark.slow
def test_long_context_prefill_and_steps(full):
    w, wd, orc = full
    wl = synth.WORKLOADS["long_context"]
    p = synth.make_prompt(wl, seed=0)
    dec = Decoder(SH, wd, max_seq=wl.max_seq)
    res = H.teacher_forced(dec, orc.clone(), p, 2)
    H.assert_step_parity(res, "long_context")
    _report("long_context", res)


def test_branching_batch(full):
    """The branching workload at full shape: one 415-position prefill cloned into 64 streams,
    each fed its own forced first token, stepped in lockstep as one batch.  Every stream's
    logits of the first lockstep step are checked against its own oracle clone, then 8
    streams spread over the batch (first, last, and both ends of each half) for 4 more steps
    with the tokens the GPU chose fed to their oracles ("Qwen3ASR ncnn多平台移植" §5: a clone
    decodes exactly like its source context)."""
    w, wd, orc = full
    wl = synth.WORKLOADS["branching_b64"]
    p = synth.make_prompt(wl, seed=0)
    src = Decoder(SH, wd, max_seq=wl.max_seq)
    src.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    o_src = orc.clone(); o_src.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    n = wl.batch
    branches = [src.clone() for _ in range(n)]
    toks = synth.make_tokens(SH.vocab, n, seed=0).numpy()
    follow = [0, 1, 15, 16, 31, 32, 62, 63]
    obr = {}
    lb = torch.empty(n, SH.vocab, device="cuda")
    am = Decoder.decode_step_batch(branches, toks, logits=lb)
    got = lb.cpu().numpy()
    assert np.array_equal(am, got.argmax(axis=1))
    for i in range(n):
        o = o_src.clone()
        z = o.decode_step(int(toks[i]))
        ok, m = oracle.parity_gate(got[i], z, H.COS_MIN, H.REL_BOUND)
        assert ok, (0, i, m)
        if i in follow:
            obr[i] = o
    toks = am
    for step in range(1, 5):
        am = Decoder.decode_step_batch(branches, toks, logits=lb)
        got = lb.cpu().numpy()
        assert np.array_equal(am, got.argmax(axis=1))
        for i in follow:
            z = obr[i].decode_step(int(toks[i]))
            ok, m = oracle.parity_gate(got[i], z, H.COS_MIN, H.REL_BOUND)
            assert ok, (step, i, m)
        toks = am
    assert all(b.position == wl.n_prompt + 5 for b in branches)
    hist = branches[37].read_history()
    assert np.array_equal(hist[:wl.n_prompt], src.read_history())


def _bf16_to_f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_kv_slots_full_shape(full):
    """KV slots of the 64-position workload after the prefill and 4 decode steps, every layer,
    against the oracle's float64 cache (the oracle's order: [position, kv head, dim]).

    Bounds, per layer, relative to that layer's max|ref|:
      * layer 0: 2^-8 (one bf16 ulp at the maximum).  The slot holds bf16(k); the GPU's k
        differs from the oracle's by the bf16 rounding of the normalised input row (the
        prefill's GEMM operand, 2^-9 relative per element, averaging out over 1024 terms)
        plus the store's half ulp.
      * every layer: 1e-2, the logits gate's bound; the residual stream carries the earlier
        layers' rounding forward, so deep layers drift as the logits do.
    Slots past the last written position stay zero."""
    w, wd, orc = full
    wl = synth.WORKLOADS["funasr_nano_short"]
    p = synth.make_prompt(wl, seed=0)
    steps = 4
    dec = Decoder(SH, wd, max_seq=wl.n_prompt + steps + 4)
    o = orc.clone()
    z = o.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    dec.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    for _ in range(steps):
        t = oracle.greedy_argmax(z)
        z = o.decode_step(t)
        dec.decode_step(t)
    n = wl.n_prompt + steps
    worst = []
    for layer in range(SH.n_layers):
        for kind, ref in ((0, o.k_cache[layer]), (1, o.v_cache[layer])):
            got = _bf16_to_f64(dec.read_kv(layer, kind, 0, n + 4))
            r = np.transpose(ref, (1, 0, 2))          # [kv head, position, dim]
            assert r.shape == got[:, :n].shape
            assert not got[:, n:].any(), (layer, kind)
            rel = np.abs(got[:, :n] - r).max() / np.abs(r).max()
            worst.append((rel, layer, kind))
            assert rel <= 1e-2, (layer, kind, rel)
            if layer == 0:
                assert rel <= 2.0 ** -8, (layer, kind, rel)
    print("kv slot error / max|ref|: worst", max(worst), "layer 0", [x for x in worst if x[1] == 0])
