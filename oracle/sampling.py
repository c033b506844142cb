"""Float64 reference of the token choice after the tied lm_head: greedy, or sampling
with temperature, top-k, top-p and repetition penalty.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code imports it.

What it follows: "Qwen3ASR ncnn多平台移植" section 1 lists greedy decoding, temperature,
top-k, top-p and repetition penalty as the generation options of its context, section 2
puts sampling and the repetition penalty in one module, and section 6 makes greedy
(temperature 0, no sampling) the default while keeping the other four for
non-deterministic experiments.  The page names the options but does not define them, so
this module takes the plainest reading of each, in the usual processing order:

  1. repetition penalty r over the distinct ids of the context's history (prompt ids and
     generated tokens): a positive logit is divided by r, a non-positive one multiplied
     by r (r = 1 leaves the logits unchanged);
  2. temperature T: logits divided by T; T = 0 means greedy (argmax, lowest index on
     ties) and nothing below applies;
  3. top-k (k <= 0 or k >= V: off): keep the logits >= the k-th largest (ties kept);
  4. top-p (p >= 1: off): with probabilities softmax over the kept logits, keep a token
     when the total probability of the tokens strictly more probable than it is < p
     (the most probable always stays; ties kept);
  5. the draw: u in [0, 1) from the counter-based generator below; the token is the
     smallest kept id j with  sum_{kept i <= j} p_i  >  u * sum_{kept} p_i.

The generator is splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014): state += 0x9E3779B97F4A7C15, then the published
mixing function.  The draw of step `pos` under `seed` is output number pos + 1 of the
generator started at state `seed` (so a kernel computes it from (seed, pos) alone), and
u keeps its top 24 bits: u = (bits >> 40) * 2^-24, exact in float32 as in float64.
"""
from __future__ import annotations

import numpy as np

_M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def splitmix64_mix(z: int) -> int:
    """The splitmix64 output function of a 64-bit state word."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def splitmix64_outputs(seed: int, n: int) -> list:
    """The first n outputs of splitmix64 started at state `seed`."""
    x, out = seed & _M64, []
    for _ in range(n):
        x = (x + GOLDEN) & _M64
        out.append(splitmix64_mix(x))
    return out


def counter_uniform(seed: int, pos: int) -> float:
    """u in [0, 1) of decode step `pos`: output pos + 1 of splitmix64 from `seed`,
    top 24 bits."""
    bits = splitmix64_mix((seed + (pos + 1) * GOLDEN) & _M64)
    return float(bits >> 40) * 2.0 ** -24


def repetition_penalty(logits, history, penalty: float) -> np.ndarray:
    """Step 1: each distinct id of `history` has its logit divided by `penalty` if it is
    positive, else multiplied by it."""
    z = np.array(logits, dtype=np.float64)
    if penalty == 1.0:
        return z
    for i in np.unique(np.asarray(history, dtype=np.int64)):
        z[i] = z[i] / penalty if z[i] > 0 else z[i] * penalty
    return z


def top_k_mask(z, k: int) -> np.ndarray:
    """Step 3: True where the logit is >= the k-th largest (every id when k is off)."""
    z = np.asarray(z, dtype=np.float64)
    if k <= 0 or k >= z.size:
        return np.ones(z.size, dtype=bool)
    kth = np.sort(z)[::-1][k - 1]
    return z >= kth


def top_p_mask(z, keep, p: float) -> np.ndarray:
    """Step 4 over the ids already kept: True where the probability mass of the kept
    tokens strictly more probable than this one is < p."""
    keep = np.asarray(keep, dtype=bool)
    if p >= 1.0:
        return keep.copy()
    z = np.asarray(z, dtype=np.float64)
    m = z[keep].max()
    w = np.where(keep, np.exp(z - m), 0.0)
    prob = w / w.sum()
    idx = np.flatnonzero(keep)
    s = prob[idx]
    order = np.argsort(-s, kind="stable")
    sd = s[order]                                   # descending
    csum = np.concatenate(([0.0], np.cumsum(sd)))   # csum[j] = mass of sd[:j]
    first = np.searchsorted(-sd, -sd, side="left")  # first index of each value's tie group
    out = np.zeros_like(keep)
    out[idx[order]] = csum[first] < p               # mass strictly more probable < p
    return out


def sample_token(logits, history, temperature: float, top_k: int, top_p: float, penalty: float,
                 seed: int, pos: int) -> int:
    """The token of decode step `pos` (steps 1-5 above); greedy when temperature is 0."""
    z = repetition_penalty(logits, history, penalty)
    if np.isnan(z).any():
        raise FloatingPointError("NaN in logits")
    if temperature == 0.0:
        return int(np.argmax(z))
    z = z / temperature
    keep = top_k_mask(z, top_k)
    keep = top_p_mask(z, keep, top_p)
    m = z[keep].max()
    w = np.where(keep, np.exp(z - m), 0.0)
    u = counter_uniform(seed, pos)
    c = np.cumsum(w)
    j = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(j, int(np.flatnonzero(keep)[-1]))
