"""Parity at full model sizes, in the launch configurations bench.py times.

The oracle computes sampled verify rows of the full 3B-MoE (bf16 and e4m3)
and dense 4B shapes one step at a time, teacher-forced on the GPU's own
committed sequence: every row's logits must sit within 2e-2 of the oracle
row's range, every GPU argmax must equal the oracle's outside near-ties
(top-1 - top-2 < 1e-3), and the accepted length and bonus must be those the
acceptance rule gives for the GPU argmaxes.

Expert routing is a discrete choice: where the oracle's k-th and (k+1)-th
router logits of a row come within ROUTE_TIE of each other at some layer,
the GPU (whose activations differ from the oracle's by rounding) may pick the
other expert, and the row's logits then move by more than the tolerance.
Such rows are exempt from the two row checks, counted, and must stay a
minority (at most a quarter of the rows).

Tokens: bf16 KV and activation rounding move a row's logits by up to the 2e-2
row tolerance, which at these vocabulary sizes is often more than the
oracle's top-1 - top-2 margin. A token mismatch therefore also passes where
that margin is below twice the row's largest |GPU - oracle| logit difference
(the flip is explained by an error the row check already bounds); these are
counted against the same quarter.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _util import gpu_model, margin_exempt, row_tol_ok

pytestmark = pytest.mark.gpu


ROUTE_TIE = 4e-3


def _check_rows(lg, ol, route_gap, rel=2e-2):
    """Returns the number of rows that needed an exemption."""
    tie = route_gap < ROUTE_TIE if route_gap is not None else np.zeros(len(lg), bool)
    ok = row_tol_ok(lg, ol, rel)
    assert (ok | tie).all(), f"logits outside 2e-2 of the row range (rows {np.nonzero(~ok)[0].tolist()})"
    g_gpu, g_or = np.argmax(lg, -1), np.argmax(ol, -1)
    err = np.abs(lg - ol).max(-1)
    flipped = np.zeros(len(lg), bool)
    for i in np.nonzero(g_gpu != g_or)[0]:
        s = np.sort(ol[i])
        margin = float(s[-1] - s[-2])
        assert margin_exempt(ol[i]) or tie[i] or margin < 2 * err[i], \
            f"token mismatch at row {i}: oracle margin {margin:.4g} >= 2 x row error {err[i]:.4g}"
        flipped[i] = True
    return int(((~ok) & tie).sum() + flipped.sum())


def _run(wl_name, n_seq, max_batch, steps, seed_drafts):
    wl = syn.WORKLOADS[wl_name]
    cfg = wl.model
    K = wl.n_draft
    w = syn.generate_weights(cfg, 0)
    om = oracle.OracleModel(w)
    prompts = syn.make_prompts(wl, n_seq=n_seq)
    max_ctx = max(p.length for p in prompts) + steps * (K + 1) + 2 * (K + 1)
    pages = sum(-(-max_ctx // wl.page_size) for _ in prompts) + 16
    gm = gpu_model(cfg, w, page_size=wl.page_size, n_pages=pages, max_seqs=max(n_seq, max_batch), max_ctx=max_ctx,
                   max_draft=K, max_batch=max_batch)
    try:
        prefix = gm.register_prefix(prompts[0].prefix_tokens) if len(prompts[0].prefix_tokens) else -1
        caches, last = [], []
        for i, p in enumerate(prompts):
            first = gm.prefill(i, p.visual, p.tokens, prefix)
            cache = oracle.KVCache(cfg)
            lg0 = oracle.forward(om, cache, oracle.prompt_embeddings(om, p), np.arange(p.length))[-1]
            assert first == int(np.argmax(lg0)) or margin_exempt(lg0)
            caches.append(cache)
            last.append(first)
        rng = np.random.default_rng(seed_drafts)
        exempt = rows = 0
        for step in range(steps):
            d = rng.integers(0, cfg.vocab, (n_seq, K)).astype(np.int32)
            # the first draft is the GPU's own next token (row 0 does not depend on
            # the drafts), so every step accepts at least one draft
            pre = gm.debug_logits(list(range(n_seq)), d).reshape(n_seq, K + 1, cfg.vocab)
            d[:, 0] = np.argmax(pre[:, 0], -1)
            lg = gm.debug_logits(list(range(n_seq)), d).reshape(n_seq, K + 1, cfg.vocab)
            for i in range(n_seq):
                tr = {}
                ol = oracle.verify_rows(om, caches[i], last[i], d[i], tr)
                exempt += _check_rows(lg[i], ol, tr.get("route_gap"))
                rows += K + 1
            a, b = gm.verify_batch(list(range(n_seq)), d, [K] * n_seq)
            for i in range(n_seq):
                exp = oracle.accept(list(d[i]), np.argmax(lg[i], -1))
                assert (int(a[i]), int(b[i])) == exp
                assert int(a[i]) >= 1
                caches[i].truncate(caches[i].length - (K + 1) + int(a[i]) + 1)
                last[i] = int(b[i])
        assert exempt * 4 <= rows, f"{exempt} of {rows} rows needed a near-tie exemption"
    finally:
        gm.close()


def test_fullsize_moe3b_bf16_b1():
    """3B-MoE bf16, 12 layers, V = 129,280, one sequence, 4 rows per step:
    the warp tensor-core GEMV path the batch-1 benchmark times."""
    _run("moe3b_bf16_b1", n_seq=1, max_batch=1, steps=3, seed_drafts=5)


def test_fullsize_moe3b_fp8_tensor_core():
    """3B-MoE with e4m3 weights and a shared 64-token prefix, model sized for
    64 sequences (the tcgen05 path the concurrency-64 benchmark times); two
    sequences are scored (a row's arithmetic does not depend on the batch)."""
    _run("moe3b_fp8_c64", n_seq=2, max_batch=64, steps=2, seed_drafts=6)


def test_fullsize_dense4b_block_draft():
    """Dense 4B shape (36 layers, GQA 32/8, inter 9,728, V = 151,936) with one
    31-token block draft per step: the tcgen05 GEMMs and the tensor-core
    attention."""
    _run("dense4b_bf16_b1", n_seq=1, max_batch=1, steps=1, seed_drafts=7)
