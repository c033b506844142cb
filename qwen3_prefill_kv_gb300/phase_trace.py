"""Phase timeline of the persistent batch-1 decode step (the QDEC_OPT_TRACE trace).

    python -m qwen3_prefill_kv_gb300.phase_trace [--workload funasr_nano_short] [--layers 10 11]

Builds the synthetic model of the workload, prefills its prompt, runs a few greedy steps,
then records the globaltimer trace of two steps and prints, per chosen layer and phase
(QKV rows, attention units, o_proj rows, gate_up pairs, down_proj rows), the median and
maximum over the working CTAs of the time the phase's input became ready and of the time
the phase finished, in microseconds from the step's start, plus the lm_head phase and the
step's total.  Needs a GPU; reads the trace through the C ABI (qdec_read_trace).
"""
from __future__ import annotations

import argparse

import numpy as np

PHASES = ["QKV", "attn", "o_proj", "gate_up", "down"]


def summarize(tr: np.ndarray, n_layers: int, layers) -> str:
    """Text summary of one step's trace [CTAs, 11 * n_layers + 8] (globaltimer ns)."""
    tr = tr.astype(np.int64)
    start = tr[:, 10 * n_layers].min()
    end = tr[:, 10 * n_layers + 3].max()
    out = [f"step total {(end - start) / 1e3:.2f} us"]
    for l in layers:
        out.append(f"layer {l}:")
        for ph, name in enumerate(PHASES):
            rdy = tr[:, 10 * l + 2 * ph]
            dn = tr[:, 10 * l + 2 * ph + 1]
            m = (rdy > 0) & (dn > 0)
            if not m.any():
                continue
            out.append(f"  {name:8s} ready med {(np.median(rdy[m]) - start) / 1e3:8.2f} max {(rdy[m].max() - start) / 1e3:8.2f}"
                       f" | done med {(np.median(dn[m]) - start) / 1e3:8.2f} max {(dn[m].max() - start) / 1e3:8.2f}"
                       f"  (CTAs {int(m.sum())})")
    work = np.zeros(len(PHASES))
    for l in range(n_layers):
        for ph in range(len(PHASES)):
            rdy = tr[:, 10 * l + 2 * ph]
            dn = tr[:, 10 * l + 2 * ph + 1]
            m = (rdy > 0) & (dn > 0)
            if m.any():
                work[ph] += np.median(dn[m] - rdy[m]) / 1e3
    out.append("median work per phase, summed over layers (us): " +
               ", ".join(f"{n} {w:.1f}" for n, w in zip(PHASES, work)))
    lr, ld = tr[:, 10 * n_layers + 1], tr[:, 10 * n_layers + 2]
    out.append(f"lm_head ready med {(np.median(lr) - start) / 1e3:.2f} max {(lr.max() - start) / 1e3:.2f}, "
               f"done med {(np.median(ld) - start) / 1e3:.2f} max {(ld.max() - start) / 1e3:.2f}")
    return "\n".join(out)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="funasr_nano_short")
    ap.add_argument("--layers", type=int, nargs="*", default=[10, 11])
    ap.add_argument("--warm-steps", type=int, default=8)
    args = ap.parse_args()
    import torch
    from . import synth, _lib
    wl = synth.WORKLOADS[args.workload]
    sh = wl.shape
    w = synth.make_weights(sh, seed=0).to("cuda")
    p = synth.make_prompt(wl, seed=0)
    dec = _lib.Decoder(sh, w, max_seq=wl.max_seq, stream=torch.cuda.current_stream())
    dec.prefill(p.ids, p.audio.cuda(), p.audio_offset)
    for _ in range(args.warm_steps):
        dec.decode_step(-1, want_argmax=False)
    dec.set_trace(True)
    traces = []
    for _ in range(2):
        dec.decode_step(-1, want_argmax=False)
        dec.sync()
        traces.append(dec.read_trace())
    dec.set_trace(False)
    for tr in traces:
        print(summarize(tr, sh.n_layers, [l for l in args.layers if l < sh.n_layers]))
    dec.close()


if __name__ == "__main__":
    main()
