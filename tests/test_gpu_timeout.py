"""Failure detection on the GPU without a fault: every wait of the persistent decode step
is bounded, and a step whose wait runs out reports QDEC_E_TIMEOUT, leaves the context
where it was, and the next run of the same step is correct.

The test shortens the bound to one poll (QDEC_OPT_SPIN_LIMIT = 1): a step then gives up at
the first ring stage or hand-off vector that is not already there, which in a 152-CTA step
with 5 dependent phases per layer happens at once.  Nothing hangs and nothing faults: the
CTAs that gave up stop issuing copies, wait for their copies in flight with the default
bound, and exit; the host reads the step's error word."""
import pytest
import torch

import oracle
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Decoder, QdecError, DECODE_PERSISTENT

import _harness as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", ["tiny", "qwen3_06b"])
def test_wait_that_runs_out_reports_timeout_and_the_step_reruns(shape):
    sh = synth.TINY if shape == "tiny" else synth.QWEN3_06B
    w = synth.make_weights(sh, seed=0)
    orc = H.make_oracle(w)
    wd = w.to("cuda")
    wl = synth.Workload("t", sh, 12, 8, 12, 0)
    p = synth.make_prompt(wl, 0)
    T = p.ids.numel()
    dec = Decoder(sh, wd, max_seq=T + 8)
    assert dec.decode_kernel == DECODE_PERSISTENT
    logits = torch.empty(sh.vocab, device="cuda")
    z = orc.prefill(p.ids.numpy(), H.audio_f64(p), p.audio_offset)
    dec.prefill(p.ids, p.audio.cuda(), p.audio_offset, logits=logits)
    ok, m = oracle.parity_gate(logits.cpu().double().numpy(), z, H.COS_MIN, H.REL_BOUND)
    assert ok, m

    tok = oracle.greedy_argmax(z)
    dec.set_option(_lib.OPT_SPIN_LIMIT, 1)
    assert dec.get_option(_lib.OPT_SPIN_LIMIT) == 1
    timeouts = 0
    for attempt in range(4):
        try:
            dec.decode_step(tok, logits=logits)
        except QdecError as e:
            assert e.status == -6, e          # QDEC_E_TIMEOUT
            assert dec.position == T          # the failed step advanced nothing
            timeouts += 1
            continue
        # a step whose waits were all satisfied at once is a correct step: undo it by prefilling again
        dec.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    assert timeouts >= 1, "no wait ran out with a one-poll bound"

    dec.set_option(_lib.OPT_SPIN_LIMIT, 0)
    for step in range(3):
        z = orc.decode_step(tok)
        a = dec.decode_step(tok, logits=logits)
        got = logits.cpu().double().numpy()
        ok, m = oracle.parity_gate(got, z, H.COS_MIN, H.REL_BOUND)
        assert ok, (step, m)
        assert a == int(got.argmax())
        tok = oracle.greedy_argmax(z)
    assert dec.position == T + 3
    dec.sync()


def test_spin_limit_option_validation():
    w = synth.make_weights(synth.TINY, seed=0).to("cuda")
    dec = Decoder(synth.TINY, w, max_seq=16)
    with pytest.raises(QdecError):
        dec.set_option(_lib.OPT_SPIN_LIMIT, -1)
    dec.set_option(_lib.OPT_SPIN_LIMIT, 1000)
    assert dec.clone().get_option(_lib.OPT_SPIN_LIMIT) == 1000
