"""Pins of the CPU oracle against things other than itself: closed forms,
brute force on tiny inputs, special cases that reduce to textbook results,
library decodes of the storage formats, and the numbers the pages print."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synthetic as syn

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))

MICRO = syn.scaled(syn.TINY, name="micro", n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2,
                   head_dim=16, n_experts=4, top_k=2, n_shared=1, inter=32, vocab=97)


def micro_model(seed=0, gamma_std=0.0, **kw):
    cfg = syn.scaled(MICRO, **kw)
    return oracle.OracleModel(syn.generate_weights(cfg, seed, norm_gamma_std=gamma_std))


def micro_prompt(cfg, n_vis=5, n_tok=3, seed=1):
    g = np.random.Generator(np.random.PCG64(seed))
    return syn.Prompt(np.zeros(0, np.int32), g.standard_normal((n_vis, cfg.hidden)).astype(np.float32),
                      g.integers(0, cfg.vocab, n_tok).astype(np.int32), 0)


# ----------------------------------------------------------------- formats --

def test_e4m3_decode_format_points():
    d = lambda c: float(oracle.decode_e4m3(np.array([c], np.uint8))[0])
    assert d(0x7E) == 448.0            # largest finite
    assert d(0x08) == 2.0 ** -6        # smallest normal
    assert d(0x01) == 2.0 ** -9        # smallest subnormal
    assert d(0x38) == 1.0
    assert d(0xB8) == -1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_e4m3_decode_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = oracle.decode_e4m3(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~fin)
    assert np.array_equal(got[fin], ref[fin])


def test_e4m3_encode_rne_saturating():
    codes = np.arange(127, dtype=np.uint8)
    vals = oracle.decode_e4m3(codes)
    assert np.array_equal(syn.f32_to_e4m3(vals), codes)          # exact values round-trip
    assert np.array_equal(syn.f32_to_e4m3(-vals[1:]), codes[1:] | 0x80)
    mids = ((vals[1:-1].astype(np.float64) + vals[2:]) / 2).astype(np.float32)
    enc = syn.f32_to_e4m3(mids)
    assert np.all(enc % 2 == 0)                                   # ties to even code
    assert syn.f32_to_e4m3(np.array([1e6], np.float32))[0] == 0x7E  # saturate
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(20000).astype(np.float32) * 50
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(syn.f32_to_e4m3(x), ref)


def test_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(1).standard_normal(50000).astype(np.float32) * 3
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(syn.f32_to_bf16_bits(x), ref)
    assert np.array_equal(oracle.decode_bf16(ref), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


# ------------------------------------------------------------------ layers --

def test_rmsnorm_closed_form():
    c, eps = 3.0, 1e-6
    g = np.linspace(0.5, 1.5, 8).astype(np.float32)
    y = oracle.rms_norm(np.full((1, 8), c, np.float32), g, eps)
    np.testing.assert_allclose(y[0], g * c / math.sqrt(c * c + eps), rtol=1e-6)
    x = np.random.default_rng(2).standard_normal((4, 32)).astype(np.float32)
    y = oracle.rms_norm(x, np.ones(32, np.float32), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-5)
    np.testing.assert_allclose(oracle.rms_norm(7 * x, np.ones(32, np.float32), 0.0), y, rtol=1e-5)


def test_rope_identity_and_complex_form():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 2, 16)).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope(x[:1], np.array([0]), 1e4), x[:1])
    pos = np.array([0, 1, 5, 17, 300, 4999])
    y = oracle.rope(x, pos, 1e4)
    # independent formulation: pair (x_i, x_{i+d/2}) as a complex number times e^{i p w_i}
    z = x[..., :8].astype(np.complex128) + 1j * x[..., 8:]
    w = 1e4 ** (-np.arange(8) * 2.0 / 16)
    zr = z * np.exp(1j * pos[:, None, None] * w[None, None, :])
    np.testing.assert_allclose(y[..., :8], zr.real, atol=2e-5)
    np.testing.assert_allclose(y[..., 8:], zr.imag, atol=2e-5)


def test_rope_relative_position():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, 32)).astype(np.float32)
    k = rng.standard_normal((1, 1, 32)).astype(np.float32)
    dots = []
    for p, pp in [(10, 3), (107, 100), (1007, 1000)]:
        dots.append(float(np.sum(oracle.rope(q, [p], 1e4) * oracle.rope(k, [pp], 1e4))))
    np.testing.assert_allclose(dots, dots[0], rtol=2e-4, atol=2e-4)


def _attn_python(q, k, v, qpos, n_kv):
    """Brute force with Python loops and math.exp (tiny inputs only)."""
    n, hq, d = q.shape
    out = np.zeros_like(q, dtype=np.float64)
    for i in range(n):
        for h in range(hq):
            kv = h * n_kv // hq
            s = [sum(float(q[i, h, t]) * float(k[c, kv, t]) for t in range(d)) / math.sqrt(d)
                 for c in range(qpos[i] + 1)]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            z = sum(e)
            for c in range(len(e)):
                out[i, h] += e[c] / z * v[c, kv].astype(np.float64)
    return out


def test_attention_brute_force_gqa():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 4, 8)).astype(np.float32)
    k = rng.standard_normal((7, 2, 8)).astype(np.float32)
    v = rng.standard_normal((7, 2, 8)).astype(np.float32)
    qpos = np.array([4, 5, 6])
    got = oracle.attention_rows(q, k, v, qpos, 2)
    np.testing.assert_allclose(got, _attn_python(q, k, v, qpos, 2), atol=1e-5)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, 1, 8)).astype(np.float32)
    q = rng.standard_normal((1, 3, 8)).astype(np.float32)
    k = rng.standard_normal((1, 1, 8)).astype(np.float32)
    # one cached key -> output is its value, for every head sharing it
    np.testing.assert_allclose(oracle.attention_rows(q, k, v, [0], 1), np.repeat(v, 3, axis=1), rtol=1e-6)
    # zero query -> uniform weights -> mean of the visible values
    vv = rng.standard_normal((5, 1, 8)).astype(np.float32)
    kk = rng.standard_normal((5, 1, 8)).astype(np.float32)
    o = oracle.attention_rows(np.zeros((1, 1, 8), np.float32), kk, vv, [3], 1)
    np.testing.assert_allclose(o[0, 0], vv[:4, 0].mean(0), rtol=1e-5, atol=1e-6)


def test_router_topk_order_and_ties():
    u = np.ones((1, 4), np.float32)
    w = np.array([[1, 0, 0, 0], [2, 0, 0, 0], [2, 0, 0, 0], [0.5, 0, 0, 0]], np.float32)
    ids, wts = oracle.route(u, w, 3)
    assert ids.tolist() == [[1, 2, 0]]                         # tie 1/2 -> lower id first
    e = np.exp(np.array([1, 2, 2, 0.5]) - 2)
    np.testing.assert_allclose(wts[0], (e / e.sum())[[1, 2, 0]], rtol=1e-6)


def _ffn_python(cfg, L, u):
    """Per-token loop with an explicit softmax and top-k selection."""
    out = np.zeros((u.shape[0], cfg.hidden))
    silu = lambda z: z / (1 + np.exp(-z))
    f = lambda e, x: L["w_down"][e].astype(np.float64) @ (
        silu(L["w_gate"][e].astype(np.float64) @ x) * (L["w_up"][e].astype(np.float64) @ x))
    for i, x in enumerate(u.astype(np.float64)):
        if cfg.n_experts:
            lg = L["w_router"].astype(np.float64) @ x
            p = np.exp(lg - lg.max()); p /= p.sum()
            chosen = sorted(range(cfg.n_experts), key=lambda e: (-p[e], e))[:cfg.top_k]
            for e in chosen:
                out[i] += p[e] * f(e, x)
        for s in range(cfg.n_shared):
            out[i] += f(cfg.n_experts + s, x)
    return out


@pytest.mark.parametrize("kw", [dict(), dict(n_experts=4, top_k=4), dict(n_experts=0, top_k=0, n_shared=1)])
def test_moe_ffn_brute_force(kw):
    m = micro_model(**kw)
    u = np.random.default_rng(7).standard_normal((5, m.cfg.hidden)).astype(np.float32)
    got = oracle.moe_ffn(m.cfg, m.layers[0], u)
    np.testing.assert_allclose(got, _ffn_python(m.cfg, m.layers[0], u), atol=2e-6)


def test_single_expert_top1_is_dense_swiglu():
    m1 = micro_model(n_experts=1, top_k=1, n_shared=0)
    md = micro_model(n_experts=0, top_k=0, n_shared=1)
    # both draw expert 0 from the same stream: routed with p = 1 equals dense
    L1, Ld = m1.layers[0], md.layers[0]
    np.testing.assert_array_equal(L1["w_gate"], Ld["w_gate"])
    u = np.random.default_rng(8).standard_normal((3, m1.cfg.hidden)).astype(np.float32)
    np.testing.assert_allclose(oracle.moe_ffn(m1.cfg, L1, u), oracle.moe_ffn(md.cfg, Ld, u), rtol=1e-6)


def test_zero_blocks_reduce_to_norm_head():
    m = micro_model()
    for L in m.layers:
        for k in ("w_qkv", "w_o", "w_down"):
            L[k] = np.zeros_like(L[k])
    p = micro_prompt(m.cfg)
    x = oracle.prompt_embeddings(m, p)
    lg = oracle.brute_force_logits(m, x)
    ref = oracle.rms_norm(x[-1:], m.final_norm, m.cfg.rms_eps) @ m.lm_head.T
    np.testing.assert_allclose(lg, ref[0], rtol=1e-5, atol=1e-6)


def test_causality():
    m = micro_model()
    p = micro_prompt(m.cfg, n_vis=6, n_tok=4)
    x = oracle.prompt_embeddings(m, p)
    a = oracle.forward(m, oracle.KVCache(m.cfg), x, np.arange(len(x)))
    x2 = x.copy(); x2[-1] += 1.0
    b = oracle.forward(m, oracle.KVCache(m.cfg), x2, np.arange(len(x)))
    np.testing.assert_array_equal(a[:-1], b[:-1])
    assert not np.allclose(a[-1], b[-1])


# --------------------------------------------------------- decode pins ----

def test_cached_decode_matches_brute_force():
    """P4: logits of cached token-by-token decode == full recompute without a cache."""
    m = micro_model(gamma_std=0.1)
    p = micro_prompt(m.cfg)
    toks, logits = oracle.greedy_decode(m, p, 12, return_logits=True)
    x = oracle.prompt_embeddings(m, p)
    for i in range(len(toks)):
        rows = np.concatenate([x, m.tok_embed[toks[:i]]]) if i else x
        np.testing.assert_allclose(oracle.brute_force_logits(m, rows), logits[i], atol=1e-5)
    tf = oracle.teacher_forced_logits(m, p, toks)
    np.testing.assert_allclose(tf, logits, atol=1e-5)
    assert np.array_equal(np.argmax(tf, -1), toks)


def test_accept_rule():
    g = [5, 6, 7, 8]
    assert oracle.accept([5, 6, 7], g) == (3, 8)      # all accepted, bonus after the last
    assert oracle.accept([5, 9, 7], g) == (1, 6)      # first divergence at draft 2
    assert oracle.accept([1, 6, 7], g) == (0, 5)      # wrong first draft: one token
    assert oracle.accept([], [4]) == (0, 4)           # no drafts = greedy step


@pytest.mark.parametrize("k", [1, 3, 31])
@pytest.mark.parametrize("mode", ["random", "correct", "wrong", "iid"])
def test_spec_equals_greedy(k, mode):
    """P1-P3: speculative output == greedy output for any drafts; all-correct
    drafts accept m every step; all-wrong drafts commit one token per step."""
    m = micro_model(seed=11)
    p = micro_prompt(m.cfg, seed=12)
    n = 40
    ref = oracle.greedy_decode(m, p, n)
    rng = np.random.default_rng(13)
    drafter = syn.Drafter("iid", 0.6, m.cfg.vocab, seed=14)

    def propose(nc, mm, step):
        if mode == "correct":
            return ref[nc:nc + mm]
        if mode == "wrong":
            return [(int(t) + 1) % m.cfg.vocab for t in ref[nc:nc + mm]]
        if mode == "random":
            return rng.integers(0, m.cfg.vocab, mm)
        return drafter.propose(ref, nc, mm, 0, step)

    toks, steps = oracle.spec_decode(m, p, n, k, propose)
    assert np.array_equal(toks, ref)
    if mode == "correct":
        assert all(a == mm for a, _, mm in steps)
        assert len(steps) == math.ceil((n - 1) / (k + 1))
    if mode == "wrong":
        assert all(a == 0 for a, _, _ in steps) and len(steps) == n - 1


def test_drafter_statistics_iid():
    """P5: E[a] = sum_i q^i for i.i.d. drafts (99% interval over 4000 steps)."""
    V, k, q, steps = 1024, 3, 0.576, 4000
    ref = np.random.default_rng(15).integers(0, V, steps * (k + 1) + 8)
    d = syn.Drafter("iid", q, V, seed=16)
    acc = []
    for s in range(steps):
        n = 1 + s * (k + 1)
        dr = d.propose(ref, n, k, 0, s)
        acc.append(oracle.accept(dr, ref[n:n + k + 1])[0])
    acc = np.array(acc, float)
    mu = syn.expected_accept_iid(q, k)
    assert abs(acc.mean() - mu) < 2.58 * acc.std() / math.sqrt(steps)
    # the pages' own accounting: acceptance = accepted / drafted, tau counts the bonus
    alpha = GOLD["acceptance_rate"]["value"]
    tau = 1 + GOLD["fastmtp_k"]["value"] * alpha
    assert round(tau, 1) == GOLD["tokens_per_verify"]["value"]


def test_drafter_statistics_geometric():
    V, k, p, steps = 151936, 31, 0.15, 3000
    ref = np.random.default_rng(17).integers(0, V, steps * (k + 1) + 40)
    d = syn.Drafter("geometric", p, V, seed=18)
    acc = []
    for s in range(steps):
        n = 1 + s * (k + 1)
        acc.append(oracle.accept(d.propose(ref, n, k, 0, s), ref[n:n + k + 1])[0])
    acc = np.array(acc, float)
    mu = syn.expected_accept_geometric(p, k)
    assert abs(mu - 5.63) < 0.01
    assert abs(acc.mean() - mu) < 2.58 * acc.std() / math.sqrt(steps)


def test_commit_pages():
    bt = [7, 3, 9, 4]
    assert oracle.commit_pages(bt, 33, 16) == ([7, 3, 9], [4])
    assert oracle.commit_pages(bt, 32, 16) == ([7, 3], [9, 4])
    assert oracle.commit_pages(bt, 32, 16, keep_pages=4) == (bt, [])
    assert oracle.commit_pages(bt, 1, 16) == ([7], [3, 9, 4])


# ------------------------------------------------------- workload shapes ---

def test_active_params_match_pages():
    """P7: the 3B-MoE shape activates ~570M parameters per token."""
    n = syn.MOE3B.active_params()
    tgt = GOLD["active_params"]["value"]
    assert abs(n - tgt) / tgt < GOLD["active_params"]["rel_tol"]
    assert syn.MOE3B.n_experts == GOLD["routed_experts"]["value"]
    assert syn.MOE3B.n_shared == GOLD["shared_experts"]["value"]
    assert syn.MOE3B.top_k == GOLD["top_k"]["value"]


def test_prompt_shapes():
    w = syn.WORKLOADS["moe3b_bf16_c32"]
    ps = syn.make_prompts(w, n_seq=64)
    nv = {len(p.visual) for p in ps}
    assert nv <= {GOLD["visual_base"]["value"] + GOLD["visual_per_tile"]["value"] * n for n in range(10)}
    assert max(nv) <= GOLD["visual_max"]["value"]
    assert all(200 <= p.out_len <= 4000 for p in ps)
    assert abs(np.mean([p.out_len for p in ps]) - GOLD["tokens_per_page"]["value"]) < 150
    assert syn.WORKLOADS["dense4b_bf16_b1"].n_draft == GOLD["block_draft"]["value"]
    # 2.57 pages/s x 1,085 tokens/page is the published 2,792 tokens/s (to rounding)
    assert abs(GOLD["pages_per_s"]["value"] * GOLD["tokens_per_page"]["value"] - GOLD["tokens_per_s"]["value"]) < 10


def test_weights_deterministic_and_thread_independent():
    a = syn.generate_weights(MICRO, 5, threads=1)
    b = syn.generate_weights(MICRO, 5, threads=4)
    assert all(np.array_equal(x, y) for x, y in zip(a.arrays, b.arrays))
    fp8 = syn.generate_weights(syn.scaled(MICRO, wdtype=syn.FP8), 5)
    w = fp8.get("w_qkv", 0)
    s = fp8.get("s_qkv", 0)
    assert w.dtype == np.uint8 and s.shape == (MICRO.qkv_rows,)
    deq = oracle.decode_e4m3(w, s)
    assert np.allclose(np.max(np.abs(deq), -1), 448 * s, rtol=1e-6)
