"""Plain float32 CPU oracle of the verify step (test infrastructure only).

Page references used below:

* [JINA] "Jina-OCR-v1: efficient document parsing with speculative decoding and
  dense verifiable rewards" -- abstract, section 1, section 3 (DeepSeekMoE
  decoder, ~570M active parameters per token), section 3.1 (draft head).
* [NEWS] "3.4B-parameter OCR model release: 2.57 pages/s on low-cost GPUs"
  (jina-ocr-v1 article) -- lossless spec decoding, KV cache of the visual
  context.
* [THREAD] "Jina AI releases jina-ocr-v1" -- 64 routed + 2 shared experts,
  top-6; greedy verification keeps the longest matching prefix; 2.7 tokens
  committed per verify.
* [E2E] "End-to-end OCR expert model architecture and acceleration principles"
  -- section 6.1 (one teacher-forced forward scores every draft position; accept
  the longest agreeing prefix left to right, the target supplies the token at
  the first divergence), section 7 (the draft / verify / append loop).
"""
from __future__ import annotations

import math
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

# --------------------------------------------------------------------------- #
# Weight decoding (storage encodings -> float32), written from the formats'
# definitions: bf16 is the top half of a binary32; OCP E4M3 has 1 sign bit, a
# 4-bit exponent with bias 7, 3 mantissa bits, subnormals at exponent 0, no
# infinities and S.1111.111 as NaN.
# --------------------------------------------------------------------------- #


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_LUT = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float32)


def decode_e4m3(codes: np.ndarray, scale: Optional[np.ndarray] = None) -> np.ndarray:
    v = _E4M3_LUT[np.asarray(codes, dtype=np.uint8)]
    if scale is not None:
        v = v * np.asarray(scale, dtype=np.float32)[..., None]
    return v.astype(np.float32)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """FP4 E2M1 codes (low 4 bits) as float32: bit 3 the sign, bits 2-1 the
    exponent with bias 1, bit 0 the mantissa; exponent 0 is subnormal
    (0 or 0.5); no infinities or NaN."""
    c = np.asarray(codes, dtype=np.uint8) & np.uint8(0xF)
    e = ((c >> 1) & 3).astype(np.int32)
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1))
    return np.where(c & 8, -mag, mag).astype(np.float32)


def decode_nvfp4(codes: np.ndarray, block_scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """NVFP4 values: each run of 16 consecutive elements along the last axis
    shares one E4M3 block scale, and the whole tensor one float32 scale:
    value = e2m1(code) * e4m3(block scale) * tensor_scale.
    codes: [..., K] (one 4-bit code per element); block_scales: [..., K/16]."""
    v = decode_e2m1(codes).astype(np.float64)
    s = decode_e4m3(block_scales).astype(np.float64)
    v = v.reshape(*v.shape[:-1], -1, 16) * s[..., None] * float(tensor_scale)
    return v.reshape(codes.shape).astype(np.float32)


def unpack_nvfp4(record: np.ndarray, rows: int, K: int):
    """The stored nvfp4 record of a [rows, K] matrix -> (codes [rows, K],
    block scale codes [rows, K/16]). Byte j of a row holds element 2j in its
    low nibble and element 2j + 1 in its high nibble; the rows' codes come
    first (rows * K / 2 bytes), then the block scales."""
    rec = np.asarray(record, dtype=np.uint8).reshape(-1)
    nc = rows * K // 2
    packed = rec[:nc].reshape(rows, K // 2)
    codes = np.empty((rows, K), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    return codes, rec[nc:nc + rows * K // 16].reshape(rows, K // 16)


class OracleModel:
    """The decoder of one model configuration with every weight decoded to
    float32 (bf16 values upcast exactly; e4m3 codes times their per-row fp32
    scale; nvfp4 codes times their block and matrix scales)."""

    def __init__(self, weights):
        cfg = weights.cfg
        self.cfg = cfg
        F32, BF16, FP8, NVFP4 = 0, 1, 2, 3

        def dec(name, layer=-1):
            i = next(k for k, (n, _, _, l) in enumerate(weights.specs)
                     if n == name and l == layer)
            _, shape, dtype, _ = weights.specs[i]
            a = weights.arrays[i]
            if int(np.prod(shape)) == 0:
                return None
            if dtype == F32:
                return np.asarray(a, dtype=np.float32)
            if dtype == BF16:
                return decode_bf16(a)
            scale = weights.get("s" + name[1:], layer)
            if dtype == NVFP4:
                rows, K = shape[-2], shape[-1]
                recs = np.asarray(a).reshape(-1, rows * K // 2 + rows * K // 16)
                mats = [decode_nvfp4(*unpack_nvfp4(r, rows, K), float(ts)) for r, ts in zip(recs, scale)]
                return np.stack(mats).reshape(shape)
            return decode_e4m3(a, scale)

        self.tok_embed = dec("tok_embed")
        self.final_norm = dec("final_norm")
        self.lm_head = dec("lm_head")
        self.layers = []
        for l in range(cfg.n_layers):
            self.layers.append(dict(
                attn_norm=dec("attn_norm", l), w_qkv=dec("w_qkv", l), w_o=dec("w_o", l),
                ffn_norm=dec("ffn_norm", l), w_router=dec("w_router", l),
                w_gate=dec("w_gate", l), w_up=dec("w_up", l), w_down=dec("w_down", l)))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> the nearest bfloat16 value (ties to the even 16-bit pattern),
    returned as float32. A bf16 value is a binary32 whose low 16 bits are zero,
    so rounding adds half an ulp of the kept part (0x7FFF, plus the kept part's
    lowest bit for ties) and clears the low half. Finite inputs only."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).reshape(np.shape(x))


class KVCache:
    """Contiguous per-layer key/value history (the oracle has no paging: paging
    only changes addresses, never values).

    The cache stores keys and values in the model's activation storage type:
    float32 for an f32 model, bfloat16 for a bf16 or e4m3-weight model (the
    KV cache is model state, held in the model's precision like its weights;
    the arithmetic on the stored values stays float32). ``kv_dtype`` ("f32" or
    "bf16") overrides that choice."""

    def __init__(self, cfg, kv_dtype: Optional[str] = None):
        self.k = [np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
                  for _ in range(cfg.n_layers)]
        self.v = [np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
                  for _ in range(cfg.n_layers)]
        if kv_dtype is None:
            kv_dtype = "f32" if cfg.wdtype == 0 else "bf16"
        assert kv_dtype in ("f32", "bf16")
        self.kv_dtype = kv_dtype

    def append(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        """Store the keys/values of new positions (rounded to the storage type)."""
        if self.kv_dtype == "bf16":
            k, v = round_bf16(k), round_bf16(v)
        self.k[layer] = np.concatenate([self.k[layer], k.astype(np.float32)])
        self.v[layer] = np.concatenate([self.v[layer], v.astype(np.float32)])

    @property
    def length(self) -> int:
        return self.k[0].shape[0]

    def truncate(self, n: int) -> None:
        """Roll back to the first ``n`` positions (rejected draft rows)."""
        self.k = [k[:n] for k in self.k]
        self.v = [v[:n] for v in self.v]

    def copy(self) -> "KVCache":
        c = KVCache.__new__(KVCache)
        c.k = list(self.k)
        c.v = list(self.v)
        c.kv_dtype = self.kv_dtype
        return c


# --------------------------------------------------------------------------- #
# Layers
# --------------------------------------------------------------------------- #

def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """z / sqrt(mean(z^2) + eps) * gamma over the last axis."""
    x = x.astype(np.float32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return (x / np.sqrt(ms + np.float32(eps))) * gamma


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half pairing: for i < d/2 the pair
    (x_i, x_{i+d/2}) is rotated by the angle p * theta^(-2i/d).
    x: [n, heads, d]; positions: [n]."""
    n, _, d = x.shape
    half = d // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]
    cos = np.cos(ang).astype(np.float32)[:, None, :]
    sin = np.sin(ang).astype(np.float32)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1).astype(np.float32)


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
                   n_kv_heads: int) -> np.ndarray:
    """Causal softmax attention. q: [n, H_q, d] at absolute positions q_pos;
    k, v: [ctx, H_kv, d] for positions 0..ctx-1. Row i attends to keys at
    positions <= q_pos[i]. Returns [n, H_q, d]."""
    n, hq, d = q.shape
    group = np.arange(hq) * n_kv_heads // hq            # q head -> kv head
    kk = k[:, group, :]                                  # [ctx, H_q, d]
    vv = v[:, group, :]
    s = np.einsum("nhd,chd->hnc", q, kk).astype(np.float32) / np.float32(math.sqrt(d))
    key_pos = np.arange(k.shape[0])
    mask = key_pos[None, :] > np.asarray(q_pos)[:, None]          # [n, ctx]
    s = np.where(mask[None, :, :], np.float32(-np.inf), s)
    s = s - np.max(s, axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / np.sum(p, axis=-1, keepdims=True, dtype=np.float32)
    return np.einsum("hnc,chd->nhd", p.astype(np.float32), vv).astype(np.float32)


def _silu(z: np.ndarray) -> np.ndarray:
    return z / (np.float32(1.0) + np.exp(-z))


def _expert(u: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """SwiGLU expert F(u) = W_d (silu(W_g u) * (W_u u)); u: [n, h]."""
    return ((_silu(u @ wg.T) * (u @ wu.T)) @ wd.T).astype(np.float32)


def route(u: np.ndarray, w_router: np.ndarray, top_k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Router of the DeepSeekMoE FFN ([JINA] section 3; [THREAD]: top-6 of 64
    routed experts): probabilities softmax(W_r u) over all experts; the top-k
    ordered by (probability desc, id asc); weights are the probabilities
    themselves (no renormalisation). Returns (ids [n, k], weights [n, k])."""
    logits = (u @ w_router.T).astype(np.float32)
    z = logits - np.max(logits, axis=-1, keepdims=True)
    p = np.exp(z)
    p = p / np.sum(p, axis=-1, keepdims=True, dtype=np.float32)
    order = np.argsort(-p, axis=-1, kind="stable")[:, :top_k]
    return order.astype(np.int32), np.take_along_axis(p, order, axis=-1).astype(np.float32)


def moe_ffn(cfg, layer: dict, u: np.ndarray) -> np.ndarray:
    """y = sum over the top-k routed experts of p_e F_e(u) + sum of the shared
    experts F_s(u). A dense model (n_experts = 0) is one shared expert."""
    n = u.shape[0]
    y = np.zeros((n, cfg.hidden), np.float32)
    E = cfg.n_experts
    if E:
        ids, wts = route(u, layer["w_router"], cfg.top_k)
        for e in range(E):
            rows, slot = np.nonzero(ids == e)
            if len(rows) == 0:
                continue
            f = _expert(u[rows], layer["w_gate"][e], layer["w_up"][e], layer["w_down"][e])
            y[rows] += wts[rows, slot][:, None] * f
    for s in range(cfg.n_shared):
        e = E + s
        y += _expert(u, layer["w_gate"][e], layer["w_up"][e], layer["w_down"][e])
    return y


def forward(m: OracleModel, cache: KVCache, x: np.ndarray, positions: np.ndarray,
            trace: Optional[dict] = None) -> np.ndarray:
    """Run rows ``x`` [n, h] at consecutive absolute ``positions`` (the first
    equal to the current cache length) through the decoder, appending their
    keys/values to ``cache``; returns float32 logits [n, vocab]. Rows attend
    causally to the cache and to earlier rows of the same call, which is the
    teacher-forced parallel scoring a verify step performs ([E2E] section 6.1).

    With ``trace`` (a dict), ``trace["route_gap"]`` receives, per row, the
    smallest gap over the layers between the k-th and (k+1)-th largest router
    logits: how close the row's expert choice came to a tie, and
    ``trace["hidden"]`` the rows' final-normed states (diagnostic outputs
    only; the arithmetic is unchanged)."""
    cfg = m.cfg
    positions = np.asarray(positions)
    assert positions[0] == cache.length
    x = x.astype(np.float32).copy()
    n = x.shape[0]
    hq, hk, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    for l, L in enumerate(m.layers):
        u = rms_norm(x, L["attn_norm"], cfg.rms_eps)
        qkv = (u @ L["w_qkv"].T).astype(np.float32)
        q = qkv[:, : hq * d].reshape(n, hq, d)
        k = qkv[:, hq * d:(hq + hk) * d].reshape(n, hk, d)
        v = qkv[:, (hq + hk) * d:].reshape(n, hk, d)
        q = rope(q, positions, cfg.rope_theta)
        k = rope(k, positions, cfg.rope_theta)
        cache.append(l, k, v)
        o = attention_rows(q, cache.k[l], cache.v[l], positions, hk)
        x = x + (o.reshape(n, hq * d) @ L["w_o"].T).astype(np.float32)
        u = rms_norm(x, L["ffn_norm"], cfg.rms_eps)
        if trace is not None and cfg.n_experts > cfg.top_k:
            rl = np.sort((u @ L["w_router"].T).astype(np.float32), axis=-1)[:, ::-1]
            gap = rl[:, cfg.top_k - 1] - rl[:, cfg.top_k]
            trace["route_gap"] = np.minimum(trace.get("route_gap", np.full(n, np.inf, np.float32)), gap)
        x = x + moe_ffn(cfg, L, u)
    u = rms_norm(x, m.final_norm, cfg.rms_eps)
    if trace is not None:
        trace["hidden"] = u                              # the LM head's input (post-norm state)
    return (u @ m.lm_head.T).astype(np.float32)


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Greedy token per row; ties go to the lowest vocabulary index."""
    return np.argmax(logits, axis=-1).astype(np.int32)   # numpy returns the first max


def prompt_embeddings(m: OracleModel, prompt) -> np.ndarray:
    """Rows of a prompt: shared-prefix token embeddings ++ visual rows ++
    instruction token embeddings."""
    parts = []
    if len(prompt.prefix_tokens):
        parts.append(m.tok_embed[np.asarray(prompt.prefix_tokens)])
    if len(prompt.visual):
        parts.append(np.asarray(prompt.visual, dtype=np.float32))
    if len(prompt.tokens):
        parts.append(m.tok_embed[np.asarray(prompt.tokens)])
    return np.concatenate(parts).astype(np.float32)


# --------------------------------------------------------------------------- #
# Decoding
# --------------------------------------------------------------------------- #

def greedy_decode(m: OracleModel, prompt, n_new: int, return_logits: bool = False):
    """Ordinary autoregressive greedy decoding with a KV cache: the prompt is
    scored once, its last row gives the first token, then one row per token.
    Exactly ``n_new`` tokens are produced (no end-of-sequence stop)."""
    cache = KVCache(m.cfg)
    x = prompt_embeddings(m, prompt)
    lg = forward(m, cache, x, np.arange(len(x)))
    toks = [int(argmax_lowest(lg[-1:])[0])]
    logits = [lg[-1]]
    while len(toks) < n_new:
        p = cache.length
        lg = forward(m, cache, m.tok_embed[[toks[-1]]], np.array([p]))
        toks.append(int(argmax_lowest(lg)[0]))
        logits.append(lg[0])
    toks = np.array(toks[:n_new], dtype=np.int32)
    return (toks, np.stack(logits[:n_new])) if return_logits else toks


def accept(drafts: Sequence[int], g: Sequence[int]) -> Tuple[int, int]:
    """Greedy acceptance ([THREAD]: keep the longest matching prefix; [E2E]
    section 6.1 and section 7: accept the agreeing prefix from the left, the
    target supplies the token at the first divergence). ``g[j]`` is the
    target's greedy token after row j (row 0 = last committed token, row j =
    draft j). Returns (a, bonus) with a = max{i : d_j = g_(j-1) for all j <= i}
    and bonus = g[a]; the step commits d_1..d_a then the bonus."""
    a = 0
    while a < len(drafts) and int(drafts[a]) == int(g[a]):
        a += 1
    return a, int(g[a])


def verify_rows(m: OracleModel, cache: KVCache, last_token: int,
                drafts: Sequence[int], trace: Optional[dict] = None) -> np.ndarray:
    """One verify forward: score rows [last_token, d_1..d_m] at the next
    positions in a single teacher-forced pass; returns logits [m+1, vocab]
    (the cache gains m+1 rows; the caller rolls back rejected ones)."""
    toks = np.array([last_token] + [int(d) for d in drafts], dtype=np.int64)
    p0 = cache.length
    return forward(m, cache, m.tok_embed[toks], np.arange(p0, p0 + len(toks)), trace)


def spec_decode(m: OracleModel, prompt, n_new: int, k: int,
                propose: Callable[[int, int, int], Sequence[int]]):
    """Greedy speculative decoding on the CPU ([E2E] section 7 loop).

    ``propose(n_committed, m, step)`` returns m drafts. Each step drafts
    m = min(k, n_new - n - 1) tokens, verifies them in one forward, commits
    d_1..d_a and the bonus token, and rolls the cache back to the committed
    length. Returns (tokens [n_new], list of (a, bonus, m) per step)."""
    cache = KVCache(m.cfg)
    x = prompt_embeddings(m, prompt)
    lg = forward(m, cache, x, np.arange(len(x)))
    toks = [int(argmax_lowest(lg[-1:])[0])]
    steps = []
    while len(toks) < n_new:
        mm = min(k, n_new - len(toks) - 1)
        d = [int(t) for t in propose(len(toks), mm, len(steps))][:mm]
        base = cache.length
        g = argmax_lowest(verify_rows(m, cache, toks[-1], d))
        a, bonus = accept(d, g)
        toks += d[:a] + [bonus]
        cache.truncate(base + a + 1)
        steps.append((a, bonus, mm))
    return np.array(toks[:n_new], dtype=np.int32), steps


def brute_force_logits(m: OracleModel, x: np.ndarray) -> np.ndarray:
    """Logits of the last row of ``x`` computed from scratch, with a fresh
    cache and every row recomputed (no reuse of earlier steps)."""
    cache = KVCache(m.cfg)
    return forward(m, cache, x, np.arange(len(x)))[-1]


def teacher_forced_logits(m: OracleModel, prompt, generated: Sequence[int]) -> np.ndarray:
    """Logits the model assigns after the prompt and after each generated
    token but the last, scored in one causal pass: row i predicts
    generated[i]. Returns [len(generated), vocab]."""
    x = prompt_embeddings(m, prompt)
    gen = np.asarray(generated, dtype=np.int64)
    rows = np.concatenate([x, m.tok_embed[gen[:-1]]]) if len(gen) > 1 else x
    cache = KVCache(m.cfg)
    lg = forward(m, cache, rows, np.arange(len(rows)))
    return lg[len(x) - 1:]


def commit_pages(block_table: Sequence[int], new_len: int, page_size: int,
                 keep_pages: int = 0) -> Tuple[List[int], List[int]]:
    """Page bookkeeping of a commit: pages wholly beyond both the committed
    length and the caller's reservation are released. Returns (kept pages,
    released pages). A page holds positions [i*P, (i+1)*P)."""
    need = max(-(-new_len // page_size), keep_pages)
    bt = [int(p) for p in block_table if p >= 0]
    return bt[:need], bt[need:]
