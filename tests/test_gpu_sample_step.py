"""The sampled verify step (spec_verify_step_sample_batch / _dev) through the
C ABI: rejection-sampling acceptance inside the model's step, the
stochastic counterpart of the greedy rule ("End-to-end OCR expert model
architecture and acceleration principles", section 6.1 and section 11 item 2).

* Rule parity: each step's (accepted, token) equals the oracle's
  oracle.sampling.rejection_sample on the step's own logits (read with
  spec_debug_logits, the same rows the step scores) and the same uniforms,
  except where the oracle's float64 decision lies within 1e-4 (relative) of
  its threshold; those are counted and must stay rare. The logits themselves
  match the oracle model's (fp32: 1e-3 max-abs; bf16: 2e-2 of the row's
  range), and the committed tokens are the accepted drafts then the token.
  Both LM-head paths: the fp32 GEMV model and a bf16 model on tcgen05.
* Law: the first token emitted after the prompt, over thousands of sampled
  steps with drafts from a drafter far from the target, is distributed as the
  oracle model's p (chi-square).
* The device-resident entry point takes the same decisions as the host one.
* K = 0 is plain sampling (one inverse-CDF draw from p_1), and a sequence's
  decisions do not depend on the other sequences of its step."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle import sampling as smp
from _util import gpu_model, row_tol_ok

pytestmark = pytest.mark.gpu

TIE = 1e-4
TINY = syn.WORKLOADS["tiny_fp32_b1"].model
MOE_SMALL = syn.scaled(syn.MOE3B, name="moe-small-bf16", n_layers=2, hidden=256, n_q_heads=2, n_kv_heads=2,
                       head_dim=128, n_experts=16, top_k=4, n_shared=2, inter=128, vocab=2048)


def _prompt(cfg, rng, n_tok=12):
    return syn.Prompt(prefix_tokens=np.zeros(0, np.int64), visual=np.zeros((0, cfg.hidden), np.float32),
                      tokens=rng.integers(0, cfg.vocab, n_tok).astype(np.int64), out_len=0)


def _oracle_rows(om, prompt, history, drafts):
    """Oracle logits of a verify step's rows: after the last committed token
    and after each draft."""
    x = oracle.prompt_embeddings(om, prompt)
    toks = np.asarray(list(history) + list(drafts), np.int64)
    rows = np.concatenate([x, om.tok_embed[toks]]).astype(np.float32)
    lg = oracle.forward(om, oracle.KVCache(om.cfg), rows, np.arange(len(rows)))
    return lg[len(x) + len(history) - 1:]


def _greedy_drafts(om, prompt, history, k, rng, hit=0.7):
    """Drafts that follow the oracle's greedy continuation with probability
    `hit` each (else a uniform token), so steps both accept and reject."""
    out = []
    for _ in range(k):
        g = int(np.argmax(_oracle_rows(om, prompt, history + out, [])[0]))
        out.append(g if rng.random() < hit else int(rng.integers(0, om.cfg.vocab)))
    return out


# temperature 0.05: the random-init models are near-flat at 1; at 0.05 the
# greedy token holds 0.25 to 0.9 of the mass, so steps both accept and reject
@pytest.mark.parametrize("cfg,temp", [(TINY, 0.05), (MOE_SMALL, 0.05)], ids=["fp32-gemv", "bf16-tcgen05"])
def test_sampled_steps_follow_the_rule(cfg, temp):
    rng = np.random.default_rng(31)
    w = syn.generate_weights(cfg, 0)
    om = oracle.OracleModel(w)
    n_seq, K = 4, 3
    gm = gpu_model(cfg, w, max_seqs=n_seq, max_ctx=256, max_draft=K, max_batch=n_seq)
    prompts = [_prompt(cfg, rng) for _ in range(n_seq)]
    hist = [[gm.prefill(s, p.visual, p.tokens)] for s, p in enumerate(prompts)]
    steps = exempt = accepted = 0
    for step in range(6):
        nd = np.array([K, K - 1, K, 0] if step % 2 else [K, K, 1, K], np.int32)
        drafts = np.zeros((n_seq, K), np.int32)
        for s in range(n_seq):
            drafts[s, :nd[s]] = _greedy_drafts(om, prompts[s], hist[s], int(nd[s]), rng)
        ua = rng.random((n_seq, K)).astype(np.float32)
        us = rng.random((n_seq, K + 1)).astype(np.float32)
        lg = gm.debug_logits(list(range(n_seq)), drafts).reshape(n_seq, K + 1, cfg.vocab)
        acc, tok = gm.verify_sample_batch(list(range(n_seq)), drafts, nd, ua, us, temp)
        for s in range(n_seq):
            k = int(nd[s])
            ref = _oracle_rows(om, prompts[s], hist[s], drafts[s, :k])
            if cfg.wdtype == syn.F32:
                assert np.abs(lg[s, :k + 1] - ref).max() < 1e-3
            else:
                assert row_tol_ok(lg[s, :k + 1], ref, 2e-2).all()
            tr = {}
            a, t = smp.rejection_sample(lg[s, :k + 1].astype(np.float64), drafts[s, :k], None,
                                        ua[s, :k].astype(np.float64), us[s, :k + 1].astype(np.float64), temp, tr)
            got = (int(acc[s]), int(tok[s]))
            assert 0 <= got[0] <= k and 0 <= got[1] < cfg.vocab
            if got != (a, t):
                m = tr["accept_margins"]
                near = min(m[: min(a, got[0]) + 1]) < TIE if m else False
                near = near or (got[0] == a and tr["sample_margin"] < TIE)
                assert near, f"step {step} seq {s}: GPU {got} vs rule {(a, t)} away from any threshold"
                exempt += 1
            hist[s] += [int(v) for v in drafts[s, :got[0]]] + [got[1]]
            assert list(gm.tokens(s)) == hist[s]
            accepted += got[0]
            steps += 1
    assert exempt * 10 <= steps, f"{exempt} of {steps} decisions within {TIE} of a threshold"
    assert 0 < accepted < 3 * steps                     # the walk both accepts and rejects


# the fp32 model scores its rows with the GEMV LM head (logits written, then
# the cooperative sampler); the bf16 one at 64 sequences with the tensor-core
# LM head, whose epilogue leaves per-tile softmax statistics instead
@pytest.mark.parametrize("cfg,temp", [(syn.scaled(TINY, name="tiny-v64", vocab=64), 1.0),
                                      (syn.scaled(MOE_SMALL, name="moe-small-v256", vocab=256), 1.0)],
                         ids=["fp32-gemv-logits", "bf16-tcgen05-tile-stats"])
def test_first_token_follows_the_target(cfg, temp):
    rng = np.random.default_rng(32)
    w = syn.generate_weights(cfg, 3)
    om = oracle.OracleModel(w)
    n, K, rounds = 64, 2, 40
    gm = gpu_model(cfg, w, max_seqs=n, max_ctx=64, max_draft=K, max_batch=n, n_pages=512)
    prompt = _prompt(cfg, rng)
    g0 = gm.prefill(0, prompt.visual, prompt.tokens)
    gm.release(0)
    p = smp.target_probs(_oracle_rows(om, prompt, [g0], [])[0], temp)
    top = int(np.argmax(p))
    first, d0s = [], []
    for _ in range(rounds):
        for s in range(n):
            assert gm.prefill(s, prompt.visual, prompt.tokens) == g0
        d = rng.integers(0, cfg.vocab, (n, K)).astype(np.int32)
        d[:, 0] = np.where(rng.random(n) < 0.5, top, d[:, 0])       # a drafter far from p
        acc, tok = gm.verify_sample_batch(list(range(n)), d, np.full(n, K, np.int32),
                                          rng.random((n, K)), rng.random((n, K + 1)), temp)
        first += list(np.where(acc >= 1, d[:, 0], tok))
        d0s += list(d[:, 0])
        for s in range(n):
            gm.release(s)
    N = len(first)
    exp = p * N
    keep = exp >= 5                                       # bins too small for the test are pooled
    obs = np.bincount(first, minlength=cfg.vocab).astype(np.float64)
    o = np.append(obs[keep], obs[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    o, e = (o, e) if e[-1] > 0 else (o[:-1], e[:-1])
    chi2 = float(((o - e) ** 2 / e).sum())
    dof = len(o) - 1
    assert chi2 < dof + 6 * np.sqrt(2 * dof), f"chi-square {chi2:.1f} with {dof} degrees of freedom"
    # the drafts' own law is far from p: the test can fail
    od = np.bincount(d0s, minlength=cfg.vocab).astype(np.float64)
    od = np.append(od[keep], od[~keep].sum())[: len(e)]
    assert float(((od - e) ** 2 / e).sum()) > 10 * (dof + 6 * np.sqrt(2 * dof))


def test_device_entry_point_matches_host():
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(33)
    cfg = MOE_SMALL
    w = syn.generate_weights(cfg, 0)
    n_seq, K = 4, 3
    models = [gpu_model(cfg, w, max_seqs=n_seq, max_ctx=256, max_draft=K, max_batch=n_seq) for _ in range(2)]
    prompts = [_prompt(cfg, rng) for _ in range(n_seq)]
    for gm in models:
        for s, p in enumerate(prompts):
            gm.prefill(s, p.visual, p.tokens)
            B.spec_reserve_seq(gm.h, s, 200)
    host, dev = models
    for step in range(4):
        drafts = rng.integers(0, cfg.vocab, (n_seq, K)).astype(np.int32)
        nd = np.array([K, 2, K, 1], np.int32)
        ua = rng.random((n_seq, K)).astype(np.float32)
        us = rng.random((n_seq, K + 1)).astype(np.float32)
        acc_h, tok_h = host.verify_sample_batch(list(range(n_seq)), drafts, nd, ua, us, 0.8)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        ids, dd, nn, uu, ss = t(np.arange(n_seq, dtype=np.int32)), t(drafts), t(nd), t(ua), t(us)
        acc_d = torch.full((n_seq,), -7, dtype=torch.int32, device="cuda")
        tok_d = torch.full((n_seq,), -7, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        B.spec_verify_step_sample_dev(dev.h, n_seq, ids, dd, nn, uu, ss, 0.8, acc_d, tok_d)
        B.spec_sync_seqs(dev.h)
        assert (acc_d.cpu().numpy() == acc_h).all() and (tok_d.cpu().numpy() == tok_h).all()
    for s in range(n_seq):
        assert list(dev.tokens(s)) == list(host.tokens(s))


@pytest.mark.parametrize("cfg,n_seq", [(TINY, 2), (MOE_SMALL, 16)], ids=["fp32-gemv", "bf16-tcgen05"])
def test_no_drafts_is_plain_sampling(cfg, n_seq):
    """K = 0: the step appends one draw from p_1 (inverse CDF with u_sample)."""
    rng = np.random.default_rng(34)
    w = syn.generate_weights(cfg, 0)
    gm = gpu_model(cfg, w, max_seqs=n_seq, max_ctx=128, max_draft=0, max_batch=n_seq)
    prompts = [_prompt(cfg, rng) for _ in range(n_seq)]
    for s, p in enumerate(prompts):
        gm.prefill(s, p.visual, p.tokens)
    ids = list(range(n_seq))
    for _ in range(3):
        us = rng.random((n_seq, 1)).astype(np.float32)
        lg = gm.debug_logits(ids, np.zeros((n_seq, 0), np.int32)).reshape(n_seq, cfg.vocab)
        acc, tok = gm.verify_sample_batch(ids, np.zeros((n_seq, 0), np.int32), np.zeros(n_seq, np.int32),
                                          np.zeros((n_seq, 0), np.float32), us, 0.05)
        assert (acc == 0).all()
        for s in ids:
            t, margin = smp.inverse_cdf(smp.target_probs(lg[s].astype(np.float64), 0.05), float(us[s, 0]))
            assert int(tok[s]) == t or margin < TIE


def test_sampled_decisions_do_not_depend_on_the_batch():
    """A sequence's (accepted, token) is the same stepped alone or with three
    others (same inputs and uniforms), on the tensor-core path."""
    rng = np.random.default_rng(35)
    cfg = MOE_SMALL
    w = syn.generate_weights(cfg, 0)
    n_seq, K = 4, 3
    prompts = [_prompt(cfg, rng) for _ in range(n_seq)]
    drafts = rng.integers(0, cfg.vocab, (3, n_seq, K)).astype(np.int32)
    ua = rng.random((3, n_seq, K)).astype(np.float32)
    us = rng.random((3, n_seq, K + 1)).astype(np.float32)
    batched = gpu_model(cfg, w, max_seqs=n_seq, max_ctx=256, max_draft=K, max_batch=n_seq)
    alone = gpu_model(cfg, w, max_seqs=n_seq, max_ctx=256, max_draft=K, max_batch=n_seq)
    for gm in (batched, alone):
        for s, p in enumerate(prompts):
            gm.prefill(s, p.visual, p.tokens)
    nd = np.full(n_seq, K, np.int32)
    for step in range(3):
        a_b, t_b = batched.verify_sample_batch(list(range(n_seq)), drafts[step], nd, ua[step], us[step], 0.05)
        for s in range(n_seq):
            a_1, t_1 = alone.verify_sample_batch([s], drafts[step, s:s + 1], nd[s:s + 1], ua[step, s:s + 1],
                                                 us[step, s:s + 1], 0.05)
            assert (int(a_1[0]), int(t_1[0])) == (int(a_b[s]), int(t_b[s])), f"step {step} sequence {s}"
    for s in range(n_seq):
        assert list(batched.tokens(s)) == list(alone.tokens(s))
