"""Pins of the FastMTP draft-head oracle (oracle/mtp.py) against what the
equations of Jina-OCR-v1 section 3.1 fix, independent of the oracle's own
code path: a zero block reduces the head to a closed form written out here;
row-by-row evaluation with a cache reproduces the one-pass grid (causality
and positions); a change to b_q moves exactly the rows on or after the
diagonal the recursion a_p^(k) = u_(p-1)^(k-1) shifts it to; rows before the
grid's start have no influence; drafting is prefix-consistent; the embedding,
output norm and LM head are the decoder's."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle import mtp

CFG = syn.TINY
N, P0, K = 12, 2, 3


@pytest.fixture(scope="module")
def head():
    m = oracle.OracleModel(syn.generate_weights(CFG, 0))
    return mtp.MtpHead(m, syn.generate_mtp_weights(CFG, 3, norm_gamma_std=0.1))


def _inputs(seed):
    rng = np.random.default_rng(seed)
    b = rng.standard_normal((N, CFG.hidden)).astype(np.float32)
    tokens = rng.integers(0, CFG.vocab, N + 1)
    return b, tokens


def _rms(x, g, eps=CFG.rms_eps):
    x = x.astype(np.float64)
    return x / np.sqrt((x * x).mean(-1, keepdims=True) + eps) * g


def test_tied_tensors_are_the_decoders(head):
    m = oracle.OracleModel(syn.generate_weights(CFG, 0))
    assert np.array_equal(head.tok_embed, m.tok_embed)
    assert np.array_equal(head.final_norm, m.final_norm)
    assert np.array_equal(head.lm_head, m.lm_head)


def test_zero_block_is_the_closed_form(head):
    """With B's matrices zero the block passes z through, so
    u_p^(k) = N_o(P [N_e(E(x_(p+1))); N_h(a_p^(k))]) with a^(1) = b, a^(k)_p = u_(p-1)^(k-1)."""
    w = dict(head.w)
    for name in ("w_qkv", "w_o", "w_gate", "w_up", "w_down"):
        w[name] = np.zeros_like(w[name])
    h0 = mtp.MtpHead.__new__(mtp.MtpHead)
    h0.cfg, h0.tok_embed, h0.final_norm, h0.lm_head, h0.w = CFG, head.tok_embed, head.final_norm, head.lm_head, w
    b, tokens = _inputs(1)
    U = mtp.grid(h0, b, tokens, P0, K)
    E, Pm = head.tok_embed.astype(np.float64), w["eh_proj"].astype(np.float64)
    ref = {}
    for k in range(1, K + 1):
        ref[k] = {}
        for p in range(P0 + k - 1, N + k - 1):
            if p + 1 > N:
                break
            a = b[p] if k == 1 else ref[k - 1][p - 1]
            z = Pm @ np.concatenate([_rms(E[tokens[p + 1]], w["enorm"]), _rms(a, w["hnorm"])])
            ref[k][p] = _rms(z, head.final_norm)
            np.testing.assert_allclose(U[k - 1][p], ref[k][p], rtol=2e-4, atol=2e-5)
    assert sorted(U[0]) == list(range(P0, N)) and sorted(U[1]) == list(range(P0 + 1, N))


def test_row_by_row_with_a_cache_equals_the_grid(head):
    b, tokens = _inputs(2)
    U = mtp.grid(head, b, tokens, P0, K)
    for k in range(1, K + 1):
        rows = sorted(U[k - 1])
        cache = None
        for r in rows:
            a = b[r:r + 1] if k == 1 else U[k - 2][r - 1][None]
            z = mtp.block_input(head, [tokens[r + 1]], a)
            y, cache = mtp.block(head, z, np.array([r]), cache, first_pos=rows[0])
            u = oracle.rms_norm(y, head.final_norm, CFG.rms_eps)[0]
            np.testing.assert_allclose(u, U[k - 1][r], rtol=1e-4, atol=1e-5)


def test_recursion_shifts_along_the_diagonal(head):
    b, tokens = _inputs(3)
    U = mtp.grid(head, b, tokens, P0, K)
    q = 6
    b2 = b.copy()
    b2[q] += 0.5
    U2 = mtp.grid(head, b2, tokens, P0, K)
    for k in range(1, K + 1):
        changed = sorted(r for r in U[k - 1] if not np.array_equal(U[k - 1][r], U2[k - 1][r]))
        assert changed == [r for r in sorted(U[k - 1]) if r >= q + k - 1], (k, changed)


def test_rows_before_the_start_do_not_matter(head):
    b, tokens = _inputs(4)
    U = mtp.grid(head, b, tokens, P0, K)
    b2, t2 = b.copy(), tokens.copy()
    b2[:P0] = 7.0
    t2[:P0 + 1] = 0                                     # tokens x_0..x_P0 are never a "next token" of a grid row
    U2 = mtp.grid(head, b2, t2, P0, K)
    for k in range(K):
        for r in U[k]:
            assert np.array_equal(U[k][r], U2[k][r])


def test_drafting_is_prefix_consistent_and_causal(head):
    b, tokens = _inputs(5)
    d3 = mtp.draft(head, b, tokens, P0, 3)
    assert mtp.draft(head, b, tokens, P0, 1) == d3[:1]
    assert mtp.draft(head, b, tokens, P0, 2) == d3[:2]
    # d_1 is the argmax of the LM head on u_p^(1), p the last row with b
    U = mtp.grid(head, b, tokens, P0, 1)
    assert d3[0] == int(np.argmax(head.lm_head @ U[0][N - 1]))
    assert all(0 <= t < CFG.vocab for t in d3)


def test_speculative_decoding_with_the_head_is_lossless(head):
    """Driving the verify loop with the head's own drafts reproduces greedy
    decoding token for token (the losslessness of greedy verification holds
    for any drafter, so a drafting bug cannot hide behind it -- but a state
    or cache bookkeeping bug in the loop would break it)."""
    m = oracle.OracleModel(syn.generate_weights(CFG, 0))
    wl = syn.WORKLOADS["tiny_fp32_b1"]
    prompt = syn.make_prompts(wl)[0]
    ref = oracle.greedy_decode(m, prompt, 24)
    toks, acc = mtp.spec_decode(m, head, prompt, 24, K)
    assert np.array_equal(toks, ref)
    assert all(0 <= a <= K for a in acc)


def test_drafts_follow_the_grid_on_teacher_forced_states(head):
    """After a prefill, the first drafts are exactly mtp.draft on the prompt's
    final-normed states and its tokens."""
    m = oracle.OracleModel(syn.generate_weights(CFG, 0))
    prompt = syn.make_prompts(syn.WORKLOADS["tiny_fp32_b1"])[0]
    cache = oracle.KVCache(CFG)
    x = oracle.prompt_embeddings(m, prompt)
    tr = {}
    lg = oracle.forward(m, cache, x, np.arange(len(x)), tr)
    first = int(np.argmax(lg[-1]))
    tokens = [0] * len(prompt.visual) + [int(t) for t in prompt.tokens] + [first]
    d = mtp.draft(head, tr["hidden"], tokens, len(prompt.visual) - 1, K)
    # the hidden rows are the LM head's inputs: they reproduce the logits
    np.testing.assert_allclose(tr["hidden"] @ m.lm_head.T, lg, rtol=1e-5, atol=1e-5)
    assert len(d) == K


def test_block_cache_is_held_in_the_storage_type():
    """The block's keys and values are stored like the decoder's cache: for a
    bf16 model they are the f32 model's keys and values rounded to bf16 (same
    weights), and a single row attends to exactly its own stored value."""
    cfg16 = syn.scaled(CFG, name="tiny-bf16", wdtype=syn.BF16)
    m16 = oracle.OracleModel(syn.generate_weights(cfg16, 0))
    h16 = mtp.MtpHead(m16, syn.generate_mtp_weights(cfg16, 3, norm_gamma_std=0.1))
    h32 = mtp.MtpHead.__new__(mtp.MtpHead)
    h32.cfg, h32.tok_embed, h32.final_norm, h32.lm_head, h32.w = CFG, h16.tok_embed, h16.final_norm, h16.lm_head, h16.w
    z = np.random.default_rng(9).standard_normal((5, CFG.hidden)).astype(np.float32)
    pos = np.arange(3, 8)
    _, (k16, v16) = mtp.block(h16, z, pos)
    _, (k32, v32) = mtp.block(h32, z, pos)
    assert np.array_equal(k16, oracle.round_bf16(k32)) and np.array_equal(v16, oracle.round_bf16(v32))
    assert not np.array_equal(k32, k16)
    assert (k16.view(np.uint32) & 0xFFFF == 0).all() and (v16.view(np.uint32) & 0xFFFF == 0).all()
    # one row: softmax over one key is 1, so the attention output is that key's stored value
    y1, (_, v1) = mtp.block(h16, z[:1], pos[:1])
    w = h16.w
    hq, hk, d = CFG.n_q_heads, CFG.n_kv_heads, CFG.head_dim
    o = np.repeat(v1.astype(np.float64), hq // hk, axis=1).reshape(1, hq * d)
    x = z[:1].astype(np.float64) + o @ w["w_o"].T.astype(np.float64)
    u = _rms(x, w["ffn_norm"])
    g = u @ w["w_gate"].T.astype(np.float64)
    x = x + ((g / (1 + np.exp(-g))) * (u @ w["w_up"].T.astype(np.float64))) @ w["w_down"].T.astype(np.float64)
    np.testing.assert_allclose(y1, x, rtol=1e-4, atol=1e-4)
