"""GPU parity of the FastMTP draft head (spec_mtp_draft) against the oracle
("Jina-OCR-v1: efficient document parsing with speculative decoding and dense
verifiable rewards", section 3.1).

The oracle follows the GPU's trajectory: its decoder states b are the
oracle's own verify-row states of the tokens the GPU committed, and every
draft is checked teacher-forced -- depth k is evaluated by the definition on
the committed tokens followed by the GPU's d_1..d_(k-1). A GPU draft must be
the oracle's argmax, or score within 1e-3 of the oracle's maximum logit (a
near-tie, counted, at most 1 in 8). Speculative decoding with the head's
drafts must equal the GPU's greedy decode token for token (lossless), also
when K changes from step to step (every depth's cache advances each call)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _util import gpu_model
from oracle import mtp

pytestmark = pytest.mark.gpu

MOE_SMALL = syn.scaled(syn.MOE3B, name="moe-small-bf16", n_layers=2, hidden=256, n_q_heads=2, n_kv_heads=2,
                       head_dim=128, n_experts=16, top_k=4, n_shared=2, inter=128, vocab=2048)
MOE_SMALL_FP8 = syn.scaled(MOE_SMALL, name="moe-small-fp8", wdtype=syn.FP8)
DENSE_SMALL = syn.scaled(syn.DENSE4B, name="dense-small-gqa", n_layers=2, hidden=256, n_q_heads=8, n_kv_heads=2,
                         head_dim=64, inter=512, vocab=2048)
TIE = 1e-3


class Track:
    """Oracle side of one sequence on the GPU's trajectory."""

    def __init__(self, om, head, prompt):
        self.om, self.head = om, head
        self.cache = oracle.KVCache(om.cfg)
        x = oracle.prompt_embeddings(om, prompt)
        tr = {}
        lg = oracle.forward(om, self.cache, x, np.arange(len(x)), tr)
        self.b = tr["hidden"]
        n_vis = len(prompt.visual)
        self.p0 = max(n_vis - 1, 0)
        self.tokens = [0] * n_vis + [int(t) for t in prompt.tokens]
        self.first_logits = lg[-1]

    def start(self, first: int):
        s = np.sort(self.first_logits)
        assert first == int(np.argmax(self.first_logits)) or s[-1] - s[-2] < TIE
        self.tokens.append(int(first))

    def check(self, d, counts):
        p = len(self.b) - 1
        for k in range(1, len(d) + 1):
            ext = self.tokens + [int(t) for t in d[:k - 1]]
            u = mtp.grid(self.head, self.b, ext, self.p0, k)[k - 1][p + k - 1]
            lg = (self.head.lm_head @ u).astype(np.float32)
            counts["drafts"] += 1
            if int(d[k - 1]) != int(np.argmax(lg)):
                gap = float(lg.max() - lg[int(d[k - 1])])
                assert gap < TIE, f"draft {k}: token {d[k - 1]} scores {gap} below the oracle's maximum"
                counts["near_tie"] += 1

    def commit(self, d, a: int, bonus: int):
        tr = {}
        base = self.cache.length
        oracle.verify_rows(self.om, self.cache, self.tokens[-1], list(d), tr)
        self.cache.truncate(base + a + 1)
        self.b = np.concatenate([self.b, tr["hidden"][: a + 1]])
        self.tokens += [int(t) for t in d[:a]] + [int(bonus)]


def _setup(cfg, n_seq, K, n_vis, n_text, seed=0, **kw):
    w = syn.generate_weights(cfg, seed)
    mw = syn.generate_mtp_weights(cfg, seed + 7, norm_gamma_std=0.1)
    om = oracle.OracleModel(w)
    head = mtp.MtpHead(om, mw)
    wl = syn.Workload("mtp", cfg, n_seq, K, "iid", 0.6, (n_vis, 0, 0), n_text, 0, (64,))
    prompts = syn.make_prompts(wl, seed=seed + 1)
    gm = gpu_model(cfg, w, max_ctx=512, max_draft=K, max_seqs=n_seq, max_batch=n_seq,
                   n_pages=48 * n_seq + 8, **kw)
    gm.attach_mtp(mw, syn.mtp_inter(cfg))
    return w, om, head, prompts, gm


def _ks(K, step):
    return [K, 1, K, 2, K][step % 5] if K > 1 else 1


def _run_parity(cfg, n_seq, K, n_vis, n_text, n_steps, seed=0):
    w, om, head, prompts, gm = _setup(cfg, n_seq, K, n_vis, n_text, seed)
    ids = list(range(n_seq))
    tracks = [Track(om, head, p) for p in prompts]
    for i, p in enumerate(prompts):
        tracks[i].start(gm.prefill(i, p.visual, p.tokens))
    counts = {"drafts": 0, "near_tie": 0}
    for step in range(n_steps):
        k = _ks(K, step)
        drafts = np.zeros((n_seq, K), np.int32)
        for i in ids:
            d = gm.mtp_draft(i, k)
            tracks[i].check(d, counts)
            drafts[i, :k] = d
        a, b = gm.verify_batch(ids, drafts, [k] * n_seq)
        for i in ids:
            tracks[i].commit(list(drafts[i, :k]), int(a[i]), int(b[i]))
    gm.close()
    assert counts["near_tie"] * 8 <= counts["drafts"], counts
    return counts


def _run_lossless(cfg, K, n_vis, n_text, n_new, seed=0):
    w, om, head, prompts, gm = _setup(cfg, 1, K, n_vis, n_text, seed)
    p = prompts[0]
    greedy = [gm.prefill(0, p.visual, p.tokens)]
    while len(greedy) < n_new:
        greedy.append(gm.verify(0, [])[1])
    gm.release(0)
    spec = [gm.prefill(0, p.visual, p.tokens)]
    accepted = []
    step = 0
    while len(spec) < n_new:
        k = min(_ks(K, step), n_new - len(spec) - 1)
        d = gm.mtp_draft(0, k) if k > 0 else []
        a, b = gm.verify(0, d)
        spec += d[:a] + [b]
        accepted.append(a)
        step += 1
    gm.close()
    assert spec[:n_new] == greedy, "speculative decoding with the head's drafts != greedy"
    return accepted


def test_mtp_drafts_tiny_fp32():
    _run_parity(syn.TINY, 1, 3, 16, 6, 10)


def test_mtp_drafts_bf16_moe():
    _run_parity(MOE_SMALL, 1, 3, 24, 6, 10)


def test_mtp_drafts_dense_gqa():
    _run_parity(DENSE_SMALL, 1, 4, 0, 9, 8)


def test_mtp_drafts_fp8_batch3_tensor_core_decoder():
    # 3 sequences x 4 rows: the decoder runs its tcgen05 path; the head reads
    # each sequence's rows of the step
    _run_parity(MOE_SMALL_FP8, 3, 3, 20, 5, 6)


def test_mtp_lossless_bf16():
    acc = _run_lossless(MOE_SMALL, 3, 24, 6, 40)
    assert len(acc) > 0


def test_mtp_lossless_fp32():
    _run_lossless(syn.TINY, 3, 16, 6, 40)


def test_mtp_reprefill_restarts_the_head():
    cfg = MOE_SMALL
    w, om, head, prompts, gm = _setup(cfg, 1, 3, 8, 5)
    p = prompts[0]
    first = gm.prefill(0, p.visual, p.tokens)
    d1 = gm.mtp_draft(0, 3)
    a, b = gm.verify(0, d1)
    gm.mtp_draft(0, 3)
    gm.release(0)
    assert gm.prefill(0, p.visual, p.tokens) == first
    assert gm.mtp_draft(0, 3) == d1
    gm.close()


def test_mtp_call_states():
    from lossless_speculative_decoding_gb300 import binding as B
    cfg = MOE_SMALL
    w, om, head, prompts, gm = _setup(cfg, 1, 3, 8, 5)
    p = prompts[0]
    gm.prefill(0, p.visual, p.tokens)
    with pytest.raises(B.SpecError) as e:
        gm.mtp_draft(0, 4)
    assert e.value.code == B.SPEC_ERR_ARG
    with pytest.raises(B.SpecError) as e:
        gm.mtp_draft(0, 0)
    assert e.value.code == B.SPEC_ERR_ARG
    d = gm.mtp_draft(0, 3)
    with pytest.raises(B.SpecError) as e:          # nothing committed since
        gm.mtp_draft(0, 3)
    assert e.value.code == B.SPEC_ERR_STATE
    gm.verify(0, d)
    gm.verify(0, [])                                # a step the head did not see
    with pytest.raises(B.SpecError) as e:
        gm.mtp_draft(0, 3)
    assert e.value.code == B.SPEC_ERR_STATE
    with pytest.raises(B.SpecError) as e:
        gm.attach_mtp(syn.generate_mtp_weights(cfg, 1), syn.mtp_inter(cfg))
    assert e.value.code == B.SPEC_ERR_STATE
    gm.release(0)
    pid = gm.register_prefix(np.arange(20, dtype=np.int32))
    gm.prefill(0, p.visual, p.tokens, prefix_id=pid)
    with pytest.raises(B.SpecError) as e:
        gm.mtp_draft(0, 3)
    assert e.value.code == B.SPEC_ERR_UNSUPPORTED
    gm.close()
