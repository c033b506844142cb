"""Per-step logits comparison (TEST INFRASTRUCTURE ONLY, see the package docstring).

"Qwen3ASR ncnn多平台移植", section 7.2 lists the per-step metrics: max abs error,
mean abs error, RMSE, mean relative error with denominator max(|ref|, 1e-6),
cosine of the full logits vectors and argmax agreement.  Section 7.1 is the
teacher-forced method these are computed under.  The relative error is reported
but not gated: near-zero reference logits inflate it (same section).
"""
from __future__ import annotations

import numpy as np


def step_metrics(cand, ref) -> dict:
    c = np.asarray(cand, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if c.shape != r.shape:
        raise ValueError("shape mismatch")
    d = c - r
    ad = np.abs(d)
    order = np.argsort(-r, kind="stable")
    gap = float(r[order[0]] - r[order[1]]) if r.size > 1 else float("inf")
    denom = np.linalg.norm(c) * np.linalg.norm(r)
    return {
        "max_abs": float(ad.max()),
        "mean_abs": float(ad.mean()),
        "rmse": float(np.sqrt(np.mean(d * d))),
        "mean_rel": float(np.mean(ad / np.maximum(np.abs(r), 1e-6))),
        "cosine": float(np.dot(c, r) / denom) if denom > 0 else float("nan"),
        "argmax_cand": int(np.argmax(c)),
        "argmax_ref": int(np.argmax(r)),
        "argmax_equal": bool(np.argmax(c) == np.argmax(r)),
        "max_abs_ref": float(np.abs(r).max()),
        "top_gap_ref": gap,
    }


def parity_gate(cand, ref, cos_min: float, rel_bound: float) -> tuple[bool, dict]:
    """True when cosine >= cos_min, max|d| <= rel_bound * max|ref|, and the
    argmax agrees wherever the reference's top-1/top-2 gap exceeds that bound.
    Where the gap is within the bound (a near tie) the candidate's pick must
    itself be a near-maximum of the reference."""
    m = step_metrics(cand, ref)
    r = np.asarray(ref, dtype=np.float64)
    bound = rel_bound * m["max_abs_ref"]
    near_tie_ok = (m["top_gap_ref"] <= bound
                   and r[m["argmax_cand"]] >= r[m["argmax_ref"]] - bound)
    ok = (m["cosine"] >= cos_min and m["max_abs"] <= bound
          and (m["argmax_equal"] or near_tie_ok))
    m["bound"] = bound
    m["pass"] = bool(ok)
    return bool(ok), m
