"""Pins of how the oracle composes its (separately pinned) primitives into a
decoder forward, of the order of a prompt's rows, and of the storage type of
its KV cache.

* Composition: a decoder layer is pre-norm attention then pre-norm FFN, each
  added to the residual stream, and the LM head reads the final-normed state
  (Jina-OCR-v1, section 3: a DeepSeekMoE decoder; the 3B-MoE shape of the
  jina-ocr-v1 release). Every norm gets its own random gain here, so feeding a
  block through the wrong norm, dropping a residual add or skipping a layer
  changes the logits; the test recomputes them from the primitives with
  Python-loop attention and FFN and checks that such mistakes are caught.
* Prompt order: shared prefix token rows, then the visual rows, then the
  instruction token rows (the OCRia-1 guide's shared prompt prefix; the
  jina-ocr-v1 article's visual tokens followed by the instruction).
* KV storage: a bf16 model keeps its cache in bf16, an f32 model in f32.
"""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn

MICRO = syn.scaled(syn.TINY, name="micro", n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2,
                   head_dim=16, n_experts=4, top_k=2, n_shared=1, inter=32, vocab=97)


def _rms(x, g, eps):
    x = x.astype(np.float64)
    return x / np.sqrt(np.mean(x * x, -1, keepdims=True) + eps) * g


def _rope(x, pos, theta):
    """Complex-number form: pair (x_i, x_(i+d/2)) times exp(i p theta^(-2i/d))."""
    d = x.shape[-1]
    h = d // 2
    z = x[..., :h].astype(np.complex128) + 1j * x[..., h:]
    w = theta ** (-np.arange(h) * 2.0 / d)
    z = z * np.exp(1j * np.asarray(pos)[:, None, None] * w[None, None, :])
    return np.concatenate([z.real, z.imag], -1)


def _attn(q, k, v, n_kv):
    """Causal attention, one loop per (row, head), rows at positions 0..n-1."""
    n, hq, d = q.shape
    out = np.zeros((n, hq, d))
    for i in range(n):
        for hh in range(hq):
            kv = hh * n_kv // hq
            s = np.array([q[i, hh] @ k[c, kv] for c in range(i + 1)]) / math.sqrt(d)
            p = np.exp(s - s.max())
            p /= p.sum()
            out[i, hh] = p @ v[: i + 1, kv]
    return out


def _ffn(cfg, L, u):
    out = np.zeros((u.shape[0], cfg.hidden))
    silu = lambda z: z / (1 + np.exp(-z))
    f = lambda e, x: L["w_down"][e].astype(np.float64) @ (
        silu(L["w_gate"][e].astype(np.float64) @ x) * (L["w_up"][e].astype(np.float64) @ x))
    for i, x in enumerate(u):
        lg = L["w_router"].astype(np.float64) @ x
        p = np.exp(lg - lg.max())
        p /= p.sum()
        for e in sorted(range(cfg.n_experts), key=lambda e: (-p[e], e))[: cfg.top_k]:
            out[i] += p[e] * f(e, x)
        for s in range(cfg.n_shared):
            out[i] += f(cfg.n_experts + s, x)
    return out


def _hand_forward(m, x, swap_norms=False, skip_attn_residual=False, layers=None):
    cfg = m.cfg
    hq, hk, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    n = len(x)
    pos = np.arange(n)
    x = x.astype(np.float64)
    for l in (range(cfg.n_layers) if layers is None else layers):
        L = m.layers[l]
        g_attn, g_ffn = (L["ffn_norm"], L["attn_norm"]) if swap_norms else (L["attn_norm"], L["ffn_norm"])
        u = _rms(x, g_attn, cfg.rms_eps)
        qkv = u @ L["w_qkv"].astype(np.float64).T
        q = _rope(qkv[:, : hq * d].reshape(n, hq, d), pos, cfg.rope_theta)
        k = _rope(qkv[:, hq * d:(hq + hk) * d].reshape(n, hk, d), pos, cfg.rope_theta)
        v = qkv[:, (hq + hk) * d:].reshape(n, hk, d)
        o = _attn(q, k, v, hk).reshape(n, hq * d) @ L["w_o"].astype(np.float64).T
        x = o if skip_attn_residual else x + o
        x = x + _ffn(cfg, L, _rms(x, g_ffn, cfg.rms_eps))
    return _rms(x, m.final_norm, cfg.rms_eps) @ m.lm_head.astype(np.float64).T


def test_forward_composition_from_primitives():
    """Two layers with distinct random gains on every norm: the oracle's
    forward equals the hand composition (pre-norm attention, residual add,
    pre-norm MoE FFN, residual add, per layer in order; final norm + LM head),
    and the plausible mistakes each move the logits far outside that match."""
    cfg = syn.scaled(MICRO, init_std=0.2)          # blocks large enough to dominate the residual
    m = oracle.OracleModel(syn.generate_weights(cfg, 21, norm_gamma_std=0.5))
    for L in m.layers:                                  # gains really differ per norm
        assert not np.allclose(L["attn_norm"], L["ffn_norm"])
    x = np.random.default_rng(22).standard_normal((7, cfg.hidden)).astype(np.float32)
    got = oracle.forward(m, oracle.KVCache(cfg), x, np.arange(7))
    ref = _hand_forward(m, x)
    tol = 1e-5 * np.max(np.abs(ref))
    np.testing.assert_allclose(got, ref, atol=tol, rtol=0)
    for wrong in (dict(swap_norms=True), dict(skip_attn_residual=True), dict(layers=[0]), dict(layers=[1, 0])):
        bad = _hand_forward(m, x, **wrong)
        assert np.max(np.abs(bad - ref)) > 1000 * tol, wrong


def test_prompt_rows_order_literal():
    """prefix token rows ++ visual rows ++ instruction token rows, literally."""
    cfg = MICRO
    m = oracle.OracleModel(syn.generate_weights(cfg, 23))
    vis = np.arange(2 * cfg.hidden, dtype=np.float32).reshape(2, cfg.hidden) / 100.0
    p = syn.Prompt(np.array([3, 1], np.int32), vis, np.array([5, 8, 2], np.int32), 0)
    rows = oracle.prompt_embeddings(m, p)
    assert rows.shape == (7, cfg.hidden)
    np.testing.assert_array_equal(rows[0], m.tok_embed[3])
    np.testing.assert_array_equal(rows[1], m.tok_embed[1])
    np.testing.assert_array_equal(rows[2:4], vis)
    np.testing.assert_array_equal(rows[4], m.tok_embed[5])
    np.testing.assert_array_equal(rows[5], m.tok_embed[8])
    np.testing.assert_array_equal(rows[6], m.tok_embed[2])
    # no prefix, no text: the visual rows alone
    q = syn.Prompt(np.zeros(0, np.int32), vis, np.zeros(0, np.int32), 0)
    np.testing.assert_array_equal(oracle.prompt_embeddings(m, q), vis)


# ------------------------------------------------------------ bf16 storage --

def test_round_bf16_format_points():
    r = lambda v: float(oracle.round_bf16(np.array([v], np.float32))[0])
    assert r(1.0) == 1.0
    assert r(1 + 2 ** -8) == 1.0                       # halfway, ties to the even pattern
    assert r(1 + 3 * 2 ** -8) == 1 + 2 ** -6           # halfway, rounds up to even
    assert r(1 + 2 ** -8 + 2 ** -20) == 1 + 2 ** -7    # just above halfway
    assert r(-(1 + 3 * 2 ** -8)) == -(1 + 2 ** -6)
    assert r(2.0 ** -130) == 2.0 ** -130                # subnormal already representable
    assert r(0.0) == 0.0


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(24).standard_normal(100000).astype(np.float32) * 7
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)


def test_kv_cache_storage_type():
    """A bf16 model stores bf16-exact keys/values; an f32 model keeps f32; with
    one cached key a row's attention output is that (stored) value."""
    cfg = syn.scaled(MICRO, wdtype=syn.BF16, n_layers=1)
    m = oracle.OracleModel(syn.generate_weights(cfg, 25))
    x = np.random.default_rng(26).standard_normal((3, cfg.hidden)).astype(np.float32)
    c = oracle.KVCache(cfg)
    assert c.kv_dtype == "bf16"
    oracle.forward(m, c, x, np.arange(3))
    for t in (c.k[0], c.v[0]):
        assert np.array_equal(oracle.round_bf16(t), t)
        assert np.any(t.view(np.uint32) & 0xFFFF) == False   # noqa: E712
    c32 = oracle.KVCache(syn.scaled(MICRO, n_layers=1))
    assert c32.kv_dtype == "f32"
    # one key: the layer's attention output is the rounded value of that key
    L = m.layers[0]
    for L_ in m.layers:
        L_["w_down"] = np.zeros_like(L_["w_down"])       # FFN adds nothing
    hq, hk, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    L["w_o"] = np.eye(cfg.hidden, hq * d, dtype=np.float32)
    row = x[:1]
    u = oracle.rms_norm(row, L["attn_norm"], cfg.rms_eps)
    v = (u @ L["w_qkv"].T)[:, (hq + hk) * d:].reshape(1, hk, d)
    kv = np.arange(hq) * hk // hq
    for vv, kind in ((oracle.round_bf16(v), "bf16"), (v, "f32")):
        o = vv[:, kv, :].reshape(1, hq * d)
        want = oracle.rms_norm(row + o, m.final_norm, cfg.rms_eps) @ m.lm_head.T
        got = oracle.forward(m, oracle.KVCache(cfg, kv_dtype=kind), row, np.arange(1))
        np.testing.assert_allclose(got, want, atol=1e-6, rtol=0)
    a = oracle.forward(m, oracle.KVCache(cfg, kv_dtype="bf16"), row, np.arange(1))
    b = oracle.forward(m, oracle.KVCache(cfg, kv_dtype="f32"), row, np.arange(1))
    assert np.max(np.abs(a - b)) > 1e-5                  # the storage type is visible
