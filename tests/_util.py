"""Shared helpers of the GPU tests: build a library model from synthetic
weights, drive a speculative run, and compare against the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synthetic as syn


def gpu_model(cfg, weights, **kw):
    from lossless_speculative_decoding_gb300.runtime import SpecModel
    return SpecModel(cfg, weights.arrays, **kw)


def run_spec(gm, seq: int, prompt, n_new: int, k: int, propose):
    """Drive spec_verify_step until n_new tokens are generated. propose(n, m, step)
    returns m drafts. Returns (tokens, per-step (drafts, a, bonus))."""
    first = gm.prefill(seq, prompt.visual, prompt.tokens)
    toks = [first]
    steps = []
    while len(toks) < n_new:
        m = min(k, n_new - len(toks) - 1)
        d = [int(x) for x in propose(len(toks), m, len(steps))][:m]
        a, b = gm.verify(seq, d)
        toks += d[:a] + [b]
        steps.append((d, a, b))
    return np.array(toks[:n_new], np.int32), steps


def margin_exempt(logits_row: np.ndarray, tol: float = 1e-3) -> bool:
    s = np.sort(logits_row)
    return float(s[-1] - s[-2]) < tol


def row_tol_ok(gpu: np.ndarray, ref: np.ndarray, rel: float) -> np.ndarray:
    """Per-row check |gpu - ref| <= rel * (max - min of the ref row)."""
    rng = ref.max(-1) - ref.min(-1)
    return np.max(np.abs(gpu - ref), -1) <= rel * rng
