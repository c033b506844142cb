"""The projector + bidirectional adaptor on the GPU against the float64 oracle
("Forward map - funasr_nano", Adaptor table; "Fun-ASR-Nano Native Runtime Implementation
Plan", Task 5), on the same bf16-rounded weights and frames, and its rows fed to the decoder
as device memory."""
import numpy as np
import pytest
import torch

import oracle
from oracle import adaptor as A
from qwen3_prefill_kv_gb300 import synth, _lib
from qwen3_prefill_kv_gb300._lib import Adaptor, Decoder

import _harness as H

pytestmark = pytest.mark.gpu
AS = synth.ADAPTOR


def _bf16(t):
    return t.to(torch.bfloat16)


@pytest.fixture(scope="module")
def adaptor_model():
    w = synth.make_adaptor_weights(AS, seed=0)
    # the GPU reads bf16 matrices and fp32 vectors; the oracle gets exactly those values
    mats = {"w1", "w2", "wq", "wk", "wv", "wo", "fc1", "fc2"}
    def gpu_side(blk):
        return {"ln1_g": blk["ln1_g"], "ln1_b": blk["ln1_b"], "ln2_g": blk["ln2_g"], "ln2_b": blk["ln2_b"],
                "wqkv": _bf16(torch.cat([blk["wq"], blk["wk"], blk["wv"]])),
                "bqkv": torch.cat([blk["bq"], blk["bk"], blk["bv"]]),
                "wo": _bf16(blk["wo"]), "bo": blk["bo"], "fc1": _bf16(blk["fc1"]), "fc1_b": blk["fc1_b"],
                "fc2": _bf16(blk["fc2"]), "fc2_b": blk["fc2_b"]}
    gw = {"w1": _bf16(w["w1"]), "b1": w["b1"], "w2": _bf16(w["w2"]), "b2": w["b2"],
          "blocks": [gpu_side(b) for b in w["blocks"]]}
    dev = {k: (v.cuda().contiguous() if torch.is_tensor(v) else [{kk: vv.cuda().contiguous() for kk, vv in b.items()}
                                                                  for b in v]) for k, v in gw.items()}
    f64 = lambda t: t.to(torch.float64).numpy()
    ow = {"w1": f64(gw["w1"]), "b1": f64(w["b1"]), "w2": f64(gw["w2"]), "b2": f64(w["b2"]), "blocks": []}
    for blk, g in zip(w["blocks"], gw["blocks"]):
        H_ = AS.hidden
        ow["blocks"].append({"ln1_g": f64(blk["ln1_g"]), "ln1_b": f64(blk["ln1_b"]),
                             "ln2_g": f64(blk["ln2_g"]), "ln2_b": f64(blk["ln2_b"]),
                             "wq": f64(g["wqkv"][:H_]), "wk": f64(g["wqkv"][H_:2 * H_]), "wv": f64(g["wqkv"][2 * H_:]),
                             "bq": f64(blk["bq"]), "bk": f64(blk["bk"]), "bv": f64(blk["bv"]),
                             "wo": f64(g["wo"]), "bo": f64(blk["bo"]), "fc1": f64(g["fc1"]), "fc1_b": f64(blk["fc1_b"]),
                             "fc2": f64(g["fc2"]), "fc2_b": f64(blk["fc2_b"])})
    return dev, ow


def _frames(T, seed):
    return _bf16(synth.make_encoder_frames(AS, T, seed=seed))


# Bound on the output rows: every projection rounds its operand rows to bf16 (2^-9 relative),
# attention rounds q, k, v and the probabilities, and the rows come out as bf16: seven bf16
# roundings on the way, each up to 2^-9 ~ 2e-3 of its values (measured on GB300: at most
# 4.0e-3 of max|ref|, cosine 0.999997).
ROW_COS, ROW_REL = 0.9999, 1e-2


@pytest.mark.parametrize("T", [183, 1, 130, 1000])
def test_adaptor_rows_match_oracle(adaptor_model, T):
    dev, ow = adaptor_model
    ad = Adaptor(AS, dev)
    fr = _frames(T, seed=T)
    ref = A.audio_rows(fr.to(torch.float64).numpy(), ow, AS.n_heads, AS.ln_eps)
    n = _lib.fake_token_len(T)
    assert ref.shape == (n, AS.hidden)
    out_dev = torch.empty(n, AS.hidden, dtype=torch.bfloat16, device="cuda")
    assert ad.run(fr.cuda(), out_dev) == n
    torch.cuda.synchronize()
    got = out_dev.cpu().to(torch.float64).numpy()
    cos = float((got * ref).sum() / np.sqrt((got * got).sum() * (ref * ref).sum()))
    rel = float(np.abs(got - ref).max() / np.abs(ref).max())
    print(f"adaptor T={T}: cos {cos:.6f} max|d|/max|ref| {rel:.4f}")
    assert cos >= ROW_COS and rel <= ROW_REL, (cos, rel)
    # host frames and host rows give the same bits
    out_host = torch.empty(n, AS.hidden, dtype=torch.bfloat16)
    ad.run(fr, out_host)
    assert torch.equal(out_host, out_dev.cpu())
    ad.close()


def test_adaptor_rows_feed_the_decoder(adaptor_model):
    """183 frames -> 23 audio rows on the device -> spliced into the 64-position prompt of the
    Fun-ASR-Nano-like workload: the decoder's prefill logits pass the parity gate against the
    oracle decoder given the same rows."""
    dev, ow = adaptor_model
    sh = synth.QWEN3_06B
    wl = synth.WORKLOADS["funasr_nano_short"]
    w = synth.make_weights(sh, seed=0)
    orc = H.make_oracle(w)
    p = synth.make_prompt(wl, seed=0)
    ad = Adaptor(AS, dev)
    rows = torch.empty(wl.n_audio, AS.hidden, dtype=torch.bfloat16, device="cuda")
    assert ad.run(_frames(183, seed=5).cuda(), rows) == wl.n_audio == 23
    dec = Decoder(sh, w.to("cuda"), max_seq=wl.n_prompt + 2)
    lg = torch.empty(sh.vocab, device="cuda")
    a = dec.prefill(p.ids, rows, p.audio_offset, logits=lg)
    z = orc.prefill(p.ids.numpy(), rows.cpu().to(torch.float64).numpy(), p.audio_offset)
    ok, m = oracle.parity_gate(lg.cpu().double().numpy(), z, H.COS_MIN, H.REL_BOUND)
    assert ok, m
    assert a == int(lg.argmax())
    ad.close()
