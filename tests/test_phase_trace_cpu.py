"""The phase-trace summarizer (qwen3_prefill_kv_gb300.phase_trace) on a synthetic trace laid
out as qdec_read_trace documents it: [10 l + 2 ph] input ready, [10 l + 2 ph + 1] phase
done, [10 NL] start, [10 NL + 1] lm_head ready, [10 NL + 2] lm_head done, [10 NL + 3] CTA
done (globaltimer ns)."""
import numpy as np

from qwen3_prefill_kv_gb300.phase_trace import summarize


def test_summary_of_a_synthetic_trace():
    NL, ctas = 2, 4
    tr = np.zeros((ctas, 11 * NL + 8), dtype=np.uint64)
    t0 = 1_000_000
    tr[:, 10 * NL] = t0 + np.arange(ctas)          # start (min = t0)
    for l in range(NL):
        for ph in range(5):
            base = t0 + (l * 5 + ph) * 2000
            tr[:, 10 * l + 2 * ph] = base + 100 * np.arange(ctas)          # ready
            tr[:, 10 * l + 2 * ph + 1] = base + 1000 + 100 * np.arange(ctas)   # done: 1 us of work
    tr[1:, 10 * 0 + 2 * 1] = 0                     # attention ran on CTA 0 only
    tr[1:, 10 * 0 + 2 * 1 + 1] = 0
    tr[:, 10 * NL + 1] = t0 + 30_000
    tr[:, 10 * NL + 2] = t0 + 40_000
    tr[:, 10 * NL + 3] = t0 + 45_000 + np.arange(ctas)
    s = summarize(tr, NL, [0])
    lines = s.splitlines()
    assert lines[0] == "step total 45.00 us"
    assert "QKV" in lines[2] and "ready med     0.15 max     0.30" in lines[2] and "(CTAs 4)" in lines[2]
    assert "attn" in lines[3] and "(CTAs 1)" in lines[3] and "ready med     2.00" in lines[3]
    assert "QKV 2.0, attn 2.0, o_proj 2.0, gate_up 2.0, down 2.0" in s   # 1 us per phase x 2 layers
    assert "lm_head ready med 30.00 max 30.00, done med 40.00 max 40.00" in s
