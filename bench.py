"""Benchmark of the Qwen3-0.6B-shape decoder hot path on one GB300 (or N replicas).

One step = one pass of the whole path over one synthetic request of the
workload: prefill of the prompt (embedding gather + audio splice, 28 layers,
tied lm_head + argmax on the last position), then the workload's greedy decode
steps at batch 1 (KV-cache decode, lm_head + argmax; the argmax is fed back on
the device).  Default workload: the Fun-ASR-Nano-like short clip, a 64-position
prompt (20 ids, 23 audio rows, 21 ids) and 64 decode steps.

value  = decode tokens/s (B = 1) over the timed steps, device-timed with CUDA
         events on the decoder's stream, inputs resident in HBM.
e2e    = the same metric end to end through the C ABI with host buffers: a
         whole request is timed (pinned host ids and audio rows copied in, the
         prefill, every decode step's argmax read back to the host and passed
         as the next token, the last logits vector copied out); value =
         generated tokens / request time.
prefill_roofline = the 4096-position prefill of the long-context workload
         (the stated tensor-core target), device-timed, against the bf16 peak.
The weights (1.19 GB) are larger than L2 (129 MB), so no L2 flush is needed
between steps.

--impl reference times the CPU oracle (float64 numpy) on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s & ms/token (B=1, Qwen3-0.6B shape), prefill tok/s, % HBM roofline"
UNIT = "tok/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="funasr_nano_short")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-long-prefill", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="streams of the branching workload (default: the workload's 64); for small profiling runs")
    ap.add_argument("--long-prefill-only", action="store_true",
                    help="time only the 4096-position prefill and print its roofline (a profiling target)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "q8b32", "q4b32"],
                    help="layer weights of the decode steps (QDEC_OPT_WEIGHTS); prefill and lm_head stay bf16")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max_over_ranks(values, world, device):
    """Element-wise maximum of `values` over the ranks (identity for one process): the
    slowest replica's times define the whole job's."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world, units_per_rank, seconds):
    """Units per second of the whole job: each of `world` replicas processed
    `units_per_rank` units, the slowest within `seconds`."""
    return world * units_per_rank / seconds


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def workload_desc(wl):
    return {"workload": wl.name, "description": wl.description, "prompt_positions": wl.n_prompt,
            "audio_rows": wl.n_audio, "audio_offset": wl.audio_offset, "decode_steps": wl.n_decode,
            "batch": wl.batch, "l2": "inputs larger than L2 (1.19 GB of bf16 weights per step), no flush"}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the decode
# kernel from an ncu capture, with the SHA-256 of the kernel's source files at that capture.
# The figure is reported only while the sources still hash to that value: any change to the
# kernel turns it into null until it is captured again.
PROFILED_DECODE_TRAFFIC = {
    "funasr_nano_short": ("cadd606c4208bef5a8cad8f8e0a5435152698ede971ea58a9ff660c9125f7c21", 1_205_231_872),
}
DECODE_KERNEL_SOURCES = ("qwen3_prefill_kv_gb300/csrc/decode_persistent.cu", "qwen3_prefill_kv_gb300/csrc/common.cuh")


def decode_sources_sha():
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_decode_traffic(workload):
    entry = PROFILED_DECODE_TRAFFIC.get(workload)
    if not entry:
        return None
    sha, traffic = entry
    return traffic if sha == decode_sources_sha() else None


def prefill_flops(shape, T):
    """Algorithmic FLOPs of a T-position prefill: the four projections on every row, the
    causal half of attention (query t attends to t + 1 keys: QK^T and PV, 2 FLOPs per MAC),
    and the tied head on the last row only."""
    H, D, F = shape.hidden, shape.head_dim, shape.ffn
    linear = 2 * T * (shape.qkv_rows * H + H * shape.n_q_heads * D + 2 * F * H + H * F)
    attn = 2 * 2 * D * shape.n_q_heads * (T * (T + 1) // 2)
    return shape.n_layers * (linear + attn) + 2 * shape.vocab * H


def time_long_prefill(w, stream, dev, reps=7, warmup=3):
    """The 4096-position prefill of the long-context workload (32 ids, 4032 audio rows, 32
    ids), replayed from its CUDA graph after the first two runs; CUDA events on the
    decoder's stream, median of `reps`.  Returns (median ms, all ms)."""
    import torch
    from qwen3_prefill_kv_gb300 import synth, _lib
    wl = synth.WORKLOADS["long_context"]
    p = synth.make_prompt(wl, seed=0)
    audio = p.audio.to(dev)
    dec = _lib.Decoder(wl.shape, w, max_seq=wl.n_prompt, stream=stream)
    for _ in range(warmup):
        dec.prefill(p.ids, audio, p.audio_offset, want_argmax=False)
    ms = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        dec.prefill(p.ids, audio, p.audio_offset, want_argmax=False)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms.append(e0.elapsed_time(e1))
    dec.sync()
    dec.close()
    return statistics.median(ms), ms


BYTES_PER_WEIGHT = {"bf16": 2.0, "q8b32": 34 / 32, "q4b32": 18 / 32}


def decode_step_bytes(shape, L, weights="bf16"):
    """Algorithmic HBM bytes of one batch-1 decode step whose KV length after the
    append is L: every weight once (embedding row only for the gather; the full
    embedding for the tied head), the KV cache read [0, L-1), the new K/V slot
    written, logits written.  `weights` is the storage of the layer matrices (codes and
    block scales for the quantized formats); norms, embedding and lm_head stay bf16."""
    H, D, F = shape.hidden, shape.head_dim, shape.ffn
    mats = shape.qkv_rows * H + H * shape.n_q_heads * D + 2 * F * H + H * F
    per_layer = mats * BYTES_PER_WEIGHT[weights] + (2 * H + 2 * D) * 2
    weights = shape.n_layers * per_layer + shape.vocab * H * 2 + H * 2 + H * 2
    kv = (L - 1) * shape.kv_bytes_per_position + shape.kv_bytes_per_position
    return weights + kv + shape.vocab * 4


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def oracle_sample(wl, n_decode, seed=0, reps=1, budget_s=None):
    """Times the CPU oracle (as it stands) on prefill + n_decode greedy steps of wl, `reps`
    times, or with a time budget until about `budget_s` seconds of oracle work (at most
    `reps` runs, at least one)."""
    import numpy as np
    import torch
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    from qwen3_prefill_kv_gb300 import synth
    w = synth.make_weights(wl.shape, seed)

    def f64(t):
        return t.to(torch.float64).numpy()
    with ThreadPoolExecutor(os.cpu_count() or 1) as ex:
        layers = [dict(zip(l.keys(), ex.map(f64, l.values()))) for l in w.layers]
        emb = f64(w.embed)
    orc = oracle.DecoderOracle(wl.shape, {"embed": emb, "final_norm": f64(w.final_norm), "layers": layers})
    p = synth.make_prompt(wl, seed)
    audio = p.audio.to(torch.float64).numpy()
    res = []
    for _ in range(reps):
        if budget_s is not None and res and sum(a + b for a, b in res) >= budget_s:
            break
        t0 = time.perf_counter()
        z = orc.prefill(p.ids.numpy(), audio, p.audio_offset)
        t1 = time.perf_counter()
        for _ in range(n_decode):
            z = orc.decode_step(oracle.greedy_argmax(z))
        t2 = time.perf_counter()
        res.append((t1 - t0, t2 - t1))
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return res, cores


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from qwen3_prefill_kv_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    n_dec = min(wl.n_decode, 64)   # the workload's decode steps (bounded for the long ones)
    res, cores = oracle_sample(wl, n_dec, reps=args.warmup + args.steps)
    timed = res[args.warmup:]
    dec_s = sum(d for _, d in timed)
    pre_s = sum(p for p, _ in timed)
    value = len(timed) * n_dec / dec_s
    sample = (f"{wl.name}: prefill of the {wl.n_prompt}-position prompt + {n_dec} greedy decode steps per step "
              f"(of the workload's {wl.n_decode}), float64 numpy oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * (dec_s + pre_s) / len(timed),
            "ms_per_token": 1e3 * dec_s / (len(timed) * n_dec),
            "prefill_tok_s": len(timed) * wl.n_prompt / pre_s, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_desc(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def batch_step_bytes(shape, Ls):
    """Algorithmic HBM bytes of one lockstep decode step over streams whose KV lengths
    after the append are Ls: every weight once for the whole batch, each stream's KV
    cache read [0, L-1) and its new slot written, each stream's logits row written."""
    H, D, F = shape.hidden, shape.head_dim, shape.ffn
    per_layer = (shape.qkv_rows * H + H * shape.n_q_heads * D + 2 * F * H + H * F + 2 * H + 2 * D) * 2
    weights = shape.n_layers * per_layer + shape.vocab * H * 2 + H * 2 + len(Ls) * H * 2
    kv = sum(L * shape.kv_bytes_per_position for L in Ls)
    return weights + kv + len(Ls) * shape.vocab * 4


def batch_step_bytes_shared(shape, Ls, P):
    """The same step when the streams are clones of one prefill sharing its first P positions
    and the batch attends that prefix once: the prefix's KV is read once for the whole batch,
    each stream's own keys [P, L) per stream."""
    H, D, F = shape.hidden, shape.head_dim, shape.ffn
    per_layer = (shape.qkv_rows * H + H * shape.n_q_heads * D + 2 * F * H + H * F + 2 * H + 2 * D) * 2
    weights = shape.n_layers * per_layer + shape.vocab * H * 2 + H * 2 + len(Ls) * H * 2
    kv = P * shape.kv_bytes_per_position + sum((L - P) * shape.kv_bytes_per_position for L in Ls)
    return weights + kv + len(Ls) * shape.vocab * 4


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    from qwen3_prefill_kv_gb300 import synth, build
    from qwen3_prefill_kv_gb300 import _lib
    build.build()
    _lib.load()
    wl = synth.WORKLOADS[args.workload]
    if args.batch and wl.batch > 1:
        import dataclasses
        wl = dataclasses.replace(wl, batch=args.batch)
    shape = wl.shape
    dev = torch.device("cuda", local_rank)
    w = synth.make_weights(shape, seed=0).to(dev)
    if args.long_prefill_only:
        stream = torch.cuda.Stream(device=dev)
        med, all_ms = time_long_prefill(w, stream, dev)
        _, bf16, peak_kind = peaks()
        fl = prefill_flops(shape, 4096)
        if rank == 0:
            print(json.dumps({"prefill_4096_ms": med, "ms_all": all_ms, "tflops": fl / (med * 1e-3) / 1e12,
                              "frac": fl / (med * 1e-3) / 1e12 / bf16, "peak_kind": peak_kind}), flush=True)
        return
    prompt = synth.make_prompt(wl, seed=rank)
    ids = prompt.ids
    audio_dev = prompt.audio.to(dev)
    stream = torch.cuda.Stream(device=dev)
    dec = _lib.Decoder(shape, w, max_seq=wl.max_seq, stream=stream)
    if args.weights != "bf16":
        if wl.batch > 1:
            raise SystemExit("--weights applies to the single-stream workloads")
        dec.set_option(_lib.OPT_WEIGHTS, {"q8b32": _lib.WEIGHTS_Q8B32, "q4b32": _lib.WEIGHTS_Q4B32}[args.weights])
    if wl.batch > 1:
        return run_ours_batch(args, wl, dec, prompt, audio_dev, stream, dev, rank, world, local_rank)

    def step_device(ev_mid=None):
        dec.prefill(ids, audio_dev, prompt.audio_offset, want_argmax=False)
        if ev_mid is not None:
            ev_mid.record(stream)
        for _ in range(wl.n_decode):
            dec.decode_step(-1, want_argmax=False)

    # warm-up (includes the one-time capture of the decode graph)
    for _ in range(args.warmup):
        step_device()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = _lib.kernel_launches()
    with ClockSampler(torch.cuda.current_device() if world == 1 else local_rank) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step_device(mids[i])
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    launches = _lib.kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    pre_ms = [s.elapsed_time(m) for s, m in zip(starts, mids)]
    dec_ms = [m.elapsed_time(e) for m, e in zip(mids, ends)]
    tot_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    clocks = clk.summary()

    # e2e through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        ids_h = ids.clone().pin_memory()
        audio_h = prompt.audio.clone().pin_memory()
        logits_h = torch.empty(shape.vocab, dtype=torch.float32).pin_memory()
        def step_host():
            tok = dec.prefill(ids_h, audio_h, prompt.audio_offset)
            for j in range(wl.n_decode):
                last = j == wl.n_decode - 1
                tok = dec.decode_step(tok, logits=logits_h if last else None)
            return tok
        for _ in range(max(1, args.warmup)):
            step_host()
        torch.cuda.synchronize(dev)
        e_req = []
        for _ in range(args.steps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            step_host()
            torch.cuda.synchronize(dev)
            e_req.append(time.perf_counter() - t0)
        # copied inside the interval, per request: the prompt ids and audio rows (host to
        # device); the argmax with the step's error word after the prefill and after every
        # decode step (8 bytes each), and the last step's logits (device to host).  Decode
        # tokens travel as kernel arguments, not as copies.
        h2d = ids.numel() * 4 + prompt.audio.numel() * 2
        d2h = (wl.n_decode + 1) * 8 + shape.vocab * 4
        e_total, = reduce_max_over_ranks([sum(e_req)], world, dev)
        e2e = {"value": whole_job_rate(world, wl.n_decode * len(e_req), e_total), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_request": 1e3 * e_total / len(e_req),
               "interval": ("whole request through the C ABI from pinned host buffers: prefill (ids and audio "
                            "copied in), then the greedy decode steps with each argmax read back to the host and "
                            "passed as the next token; value = generated tokens / interval")}

    dec_total_s = sum(dec_ms) / 1e3
    pre_total_s = sum(pre_ms) / 1e3
    dec_total_s, pre_total_s, tot = reduce_max_over_ranks([dec_total_s, pre_total_s, sum(tot_ms)], world, dev)
    tot_ms_mean = tot / args.steps
    value = whole_job_rate(world, wl.n_decode * args.steps, dec_total_s)
    hbm, bf16, peak_kind = peaks()
    # roofline of the decode step (the dominant part of the step): algorithmic bytes per
    # step averaged over the KV lengths the timed steps see, over the mean step time.
    Ls = range(wl.n_prompt + 1, wl.n_prompt + wl.n_decode + 1)
    bytes_per_token = sum(decode_step_bytes(shape, L, args.weights) for L in Ls) / len(Ls)
    t_tok = dec_total_s / (wl.n_decode * args.steps)
    achieved = bytes_per_token / t_tok / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_ms_mean, "ms_per_token": 1e3 * t_tok,
            "prefill_tok_s": whole_job_rate(world, wl.n_prompt * args.steps, pre_total_s),
            "prefill_ms": 1e3 * pre_total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init bf16 weights of the Qwen3-0.6B shape; seeded ids and audio rows)",
            "config": dict(workload_desc(wl), parallelism=f"replicas{world}", decode_weights=args.weights),
            "roofline": {"bound": "hbm",
                         "kernel": ("decode_persistent_kernel (one launch per token)" if dec.decode_kernel == 0
                                    else "decode step (graph of the CUDA-core kernels of one token)"),
                         "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "peak_kind": peak_kind,
                         "traffic": (profiled_decode_traffic(wl.name) if dec.decode_kernel == 0 else None),
                         "algorithmic_bytes_per_launch": bytes_per_token},
            "clocks": clocks, "gpu_launches": int(launches) * world,
            "e2e": e2e}
    if not args.no_long_prefill:
        # the stated prefill target: the 4096-position prompt against the bf16 tensor peak
        med, all_ms = time_long_prefill(w, stream, dev)
        med, = reduce_max_over_ranks([med], world, dev)
        fl = prefill_flops(shape, 4096)
        ach = fl / (med * 1e-3) / 1e12
        line["prefill_4096_ms"] = med
        line["prefill_roofline"] = {"bound": "tensor", "workload": "long_context prefill (4096 positions)",
                                    "flops": fl, "achieved": ach, "peak": bf16, "unit": "TFLOP/s",
                                    "frac": ach / bf16, "peak_kind": f"{peak_kind} bf16 burst",
                                    "ms_all": all_ms, "timing": "median of 7 graph replays, CUDA events"}
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        try:
            # the workload's own prefill and decode steps, repeated to about 10 s of oracle work
            res, cores = oracle_sample(wl, wl.n_decode, reps=8, budget_s=10.0)
            p_s, d_s = sum(a for a, _ in res), sum(b for _, b in res)
            line["cpu_baseline"] = {"value": len(res) * wl.n_decode / d_s, "unit": UNIT, "cores": cores,
                                    "kind": "oracle",
                                    "sample": f"{wl.name}: {len(res)} run(s) of the prefill of {wl.n_prompt} positions "
                                              f"({p_s:.2f} s) + {wl.n_decode} greedy decode steps ({d_s:.2f} s), "
                                              f"float64 numpy oracle"}
        except Exception as e:  # pragma: no cover
            line["cpu_baseline"] = {"value": None, "unit": UNIT, "cores": None, "kind": "oracle",
                                    "sample": f"failed: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dec.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_ours_batch(args, wl, dec, prompt, audio_dev, stream, dev, rank, world, local_rank):
    """Branching workload: one prefill, wl.batch clones of its state, each with its own
    seeded forced first token, then wl.n_decode lockstep decode steps of the whole batch
    (each stream's argmax fed back on the device).  value = decode tokens/s of the batch."""
    import numpy as np
    import torch
    from qwen3_prefill_kv_gb300 import synth
    from qwen3_prefill_kv_gb300._lib import Decoder
    from qwen3_prefill_kv_gb300 import _lib
    shape, n = wl.shape, wl.batch
    first = synth.make_tokens(shape.vocab, n, seed=rank).numpy()
    feedback = np.full(n, -1, dtype=np.int32)

    def step(ev_mid=None):
        dec.prefill(prompt.ids, audio_dev, prompt.audio_offset, want_argmax=False)
        br = [dec.clone() for _ in range(n)]
        if ev_mid is not None:
            ev_mid.record(stream)
        Decoder.decode_step_batch(br, first, want_argmax=False)
        for _ in range(wl.n_decode - 1):
            Decoder.decode_step_batch(br, feedback, want_argmax=False)
        return br

    def close(br):
        for b in br:
            b.close()

    for _ in range(args.warmup):
        close(step())
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    pre_ms, dec_ms = [], []
    launches = 0
    with ClockSampler(torch.cuda.current_device() if world == 1 else local_rank) as clk:
        for _ in range(args.steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            torch.cuda.synchronize(dev)
            l0 = _lib.kernel_launches()
            ev[0].record(stream)
            br = step(ev[1])
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            launches += _lib.kernel_launches() - l0
            pre_ms.append(ev[0].elapsed_time(ev[1]))
            dec_ms.append(ev[1].elapsed_time(ev[2]))
            close(br)
    clocks = clk.summary()

    e2e = None
    if not args.no_e2e:
        ids_h = prompt.ids.clone().pin_memory()
        audio_h = prompt.audio.clone().pin_memory()
        logits_h = torch.empty(n, shape.vocab, dtype=torch.float32).pin_memory()

        def step_host():
            dec.prefill(ids_h, audio_h, prompt.audio_offset)
            br = [dec.clone() for _ in range(n)]
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            toks = first
            for j in range(wl.n_decode):
                last = j == wl.n_decode - 1
                toks = Decoder.decode_step_batch(br, toks, logits=logits_h if last else None)
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
            close(br)
            return dt
        for _ in range(max(1, args.warmup)):
            step_host()
        e_dec = [step_host() for _ in range(args.steps)]
        h2d = prompt.ids.numel() * 4 + prompt.audio.numel() * 2 + wl.n_decode * n * 4
        d2h = (wl.n_decode + 1) * n * 4 + n * shape.vocab * 4
        e_total, = reduce_max_over_ranks([sum(e_dec)], world, dev)
        e2e = {"value": whole_job_rate(world, n * wl.n_decode * len(e_dec), e_total), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_lockstep": 1e3 * e_total / (wl.n_decode * len(e_dec))}

    dec_total_s = sum(dec_ms) / 1e3
    pre_total_s = sum(pre_ms) / 1e3
    tot_ms_mean = (sum(dec_ms) + sum(pre_ms)) / args.steps
    dec_total_s, pre_total_s, tot_ms_mean = reduce_max_over_ranks([dec_total_s, pre_total_s, tot_ms_mean], world, dev)
    value = whole_job_rate(world, n * wl.n_decode * args.steps, dec_total_s)
    hbm, _, peak_kind = peaks()
    t_lock = dec_total_s / (wl.n_decode * args.steps)
    bytes_per_lock = sum(batch_step_bytes(shape, [wl.n_prompt + 1 + j] * n) for j in range(wl.n_decode)) / wl.n_decode
    bytes_shared = sum(batch_step_bytes_shared(shape, [wl.n_prompt + 1 + j] * n, wl.n_prompt)
                       for j in range(wl.n_decode)) / wl.n_decode
    achieved = bytes_per_lock / t_lock / 1e9
    achieved_shared = bytes_shared / t_lock / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_ms_mean, "ms_per_lockstep": 1e3 * t_lock,
            "ms_per_token": 1e3 * t_lock / n,
            "prefill_and_clone_ms": 1e3 * pre_total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init bf16 weights of the Qwen3-0.6B shape; seeded ids, audio rows "
                    "and forced first tokens)",
            "config": dict(workload_desc(wl), parallelism=f"replicas{world}"),
            "roofline": {"bound": "hbm", "kernel": "lockstep decode step (all kernels of one batch step)",
                         "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "peak_kind": peak_kind, "traffic": None,
                         "algorithmic_bytes_per_launch": bytes_per_lock,
                         "denominator": "every stream reads its own copy of the prefix's KV",
                         "shared_prefix": {"algorithmic_bytes_per_launch": bytes_shared,
                                           "achieved": achieved_shared, "frac": achieved_shared / hbm,
                                           "denominator": "the 415-position prefix's KV read once per step"}},
            "clocks": clocks, "gpu_launches": int(launches) * world, "e2e": e2e}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dec.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
