"""Rejection-sampling verification -- the stochastic counterpart of the greedy
acceptance rule (test infrastructure only; same import rule as the rest of
this package).

Page references:

* [E2E] "End-to-end OCR expert model architecture and acceleration principles"
  -- section 6.1 (the verify step keeps the agreeing prefix and the target
  supplies the token at the first divergence; rejection sampling keeps the
  output distribution equal to the target model's own), section 11 item 2
  (speculative decoding changes latency only, not the output distribution).

The pages state the property, not the algorithm. This module takes the
plainest rule that has it, the published speculative-sampling rule: with
target distributions p_j (row j - 1 of the verify logits, softmax at
temperature tau) and the drafter's distributions q_j, walk the drafts left to
right; accept d_j when u_j * q_j(d_j) < p_j(d_j) (u_j uniform on [0, 1), i.e.
with probability min(1, p_j(d_j) / q_j(d_j))); at the first rejection draw the
appended token from the normalised residual max(0, p_j - q_j); when every
draft is accepted draw it from p_(K+1). Then the first token emitted at each
position is distributed as p exactly:
P(v) = min(p(v), q(v)) + sum_w max(0, p(w) - q(w)) * max(0, p(v) - q(v)) / S
     = p(v).

Readings of what the pages leave open:

* The random numbers are inputs: u_accept[j] for the test at draft j and
  u_sample[j] for the draw at the stopping row j (u_sample[K] for the bonus).
* A draw from weights r over the vocabulary is the inverse CDF in index
  order: the smallest v with r(0) + ... + r(v) > u * (r(0) + ... + r(V-1)).
* q = None stands for a drafter that is certain of its drafts (one-hot q_j
  at d_j, as the greedy drafters are).
* Everything here is float64; the device takes the same decisions in
  float32, so ``trace`` reports how far each decision was from its
  threshold and tests exempt decisions closer than the float32 error.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np


def target_probs(logits_row: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(logits / temperature) in float64 (max subtracted first)."""
    z = np.asarray(logits_row, np.float64) / float(temperature)
    e = np.exp(z - z.max())
    return e / e.sum()


def inverse_cdf(weights: np.ndarray, u: float) -> Tuple[int, float]:
    """Smallest v with cumsum(weights)[v] > u * sum(weights); returns (v,
    distance of u * S to the nearest bucket edge, relative to S)."""
    c = np.cumsum(np.asarray(weights, np.float64))
    s = c[-1]
    target = u * s
    v = int(np.searchsorted(c, target, side="right"))
    v = min(v, len(c) - 1)
    lo = c[v - 1] if v > 0 else 0.0
    margin = min(target - lo, c[v] - target) / s if s > 0 else 0.0
    return v, margin


def rejection_sample(logits: np.ndarray, drafts: Sequence[int], q: Optional[np.ndarray],
                     u_accept: Sequence[float], u_sample: Sequence[float], temperature: float = 1.0,
                     trace: Optional[dict] = None) -> Tuple[int, int]:
    """One sequence's verify decision under rejection sampling.

    logits: [K+1, V] target logits (row 0 after the last committed token, row j
    after draft j); drafts: K tokens; q: [K, V] drafter probabilities or None
    (one-hot at the drafts); u_accept: K uniforms; u_sample: K+1 uniforms.
    Returns (a, token): a drafts accepted, then ``token`` appended (the
    residual draw at the first rejection, or the bonus draw from row K)."""
    K = len(drafts)
    margins = []
    for j in range(K):
        p = target_probs(logits[j], temperature)
        d = int(drafts[j])
        qd = 1.0 if q is None else float(q[j][d])
        lhs, rhs = float(u_accept[j]) * qd, float(p[d])
        margins.append(abs(lhs - rhs) / max(rhs, 1e-300))
        if lhs < rhs:
            continue
        qrow = np.zeros_like(p) if q is None else np.asarray(q[j], np.float64)
        if q is None:
            qrow[d] = 1.0
        r = np.maximum(p - qrow, 0.0)
        if r.sum() <= 0.0:            # p == q: a rejection has probability zero
            r = p
        t, m = inverse_cdf(r, float(u_sample[j]))
        if trace is not None:
            trace["accept_margins"] = margins
            trace["sample_margin"] = m
        return j, t
    p = target_probs(logits[K], temperature)
    t, m = inverse_cdf(p, float(u_sample[K]))
    if trace is not None:
        trace["accept_margins"] = margins
        trace["sample_margin"] = m
    return K, t


def spec_sample_decode(m, prompt, n_new: int, K: int, propose, temperature: float, rng):
    """Speculative decoding with rejection-sampling verification (the loop of
    the end-to-end OCR explainer, section 7: draft, verify, append), the
    target's own first token drawn from its distribution too.
    ``propose(tokens, k)`` returns (drafts [k], q [k, V] or None); uniforms
    come from ``rng`` (numpy Generator): per step k acceptance uniforms, then
    k + 1 sampling uniforms. Returns the generated tokens [n_new]."""
    from .model import KVCache, forward, prompt_embeddings, verify_rows
    cache = KVCache(m.cfg)
    x = prompt_embeddings(m, prompt)
    lg = forward(m, cache, x, np.arange(len(x)))
    out = [inverse_cdf(target_probs(lg[-1], temperature), float(rng.random()))[0]]
    while len(out) < n_new:
        k = min(K, n_new - len(out) - 1)
        d, q = propose(list(out), k)
        base = cache.length
        logits = verify_rows(m, cache, out[-1], d)
        ua, us = rng.random(k), rng.random(k + 1)
        a, t = rejection_sample(logits, d, q, ua, us, temperature)
        cache.truncate(base + a + 1)
        out += [int(v) for v in d[:a]] + [int(t)]
    return np.array(out[:n_new], np.int32)
