"""FastMTP draft head: the drafter that produces the K drafts a verify step
checks (test infrastructure only; same import rule as the rest of this
package).

Page: "Jina-OCR-v1: efficient document parsing with speculative decoding and
dense verifiable rewards", section 3.1 (draft-head architecture). One draft
block applied recursively for K = 3 steps. For sequence position p and
recursion depth k, with e_p = E(x_p) the embedding of token x_p and b_p the
decoder's post-normalisation state after x_p:
    a_p^(1) = b_p,   a_p^(k) = u_(p-1)^(k-1)  (k > 1),
    z_p^(k) = P([N_e(e_(p+1)); N_h(a_p^(k))]),
    u_p^(k) = N_o(B(z_p^(k); pos = p)),   l_p^(k) = W_lm u_p^(k);
N_e, N_h normalisations, P a linear projection, B the shared dense block
(enorm, hnorm, eh_proj, mtp_block); E, N_o and W_lm are the decoder's own.

Readings of what the section leaves open:
* B is one decoder layer of the decoder's attention shape with a dense SwiGLU
  FFN (width ``synthetic.mtp_inter``): x + Attn(RMSNorm(x)), then
  + FFN(RMSNorm(.)). Its attention is causal over the rows of the same depth:
  the equations define u on a grid of (position, depth), and row p of depth k
  attends to rows <= p of depth k, at RoPE position p.
* The block's keys and values are stored like the decoder's KV cache: bf16
  for bf16 and e4m3-weight models, f32 for f32 models.
* N_e and N_h are RMSNorms with their own gains; P is [h, 2h] applied to the
  concatenation [N_e(e); N_h(a)]; b_p is the decoder's final-normed state (the
  LM head's input).
* The grid starts at the first row whose next input is a token (the last
  visual row, or row 0 without visual rows); depth k starts k - 1 rows later,
  since a_p^(k) needs row p - 1 of depth k - 1.
* Drafting after committed tokens x_0..x_(p+1) (b_0..b_p known): d_k is the
  argmax of l^(k) at row p + k - 1 of the grid evaluated on x_0..x_(p+1),
  d_1..d_(k-1) -- the equations applied to the committed sequence followed by
  the drafts made so far, every input they name teacher-forced. Ties keep the
  lowest index.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from .model import (KVCache, OracleModel, _silu, accept, argmax_lowest, attention_rows, forward, round_bf16,
                    prompt_embeddings, rms_norm, rope, verify_rows)


class MtpHead:
    """The draft head: its own tensors plus the decoder's tied embedding,
    output norm and LM head."""

    def __init__(self, m: OracleModel, w: Dict[str, np.ndarray]):
        self.cfg = m.cfg
        self.tok_embed, self.final_norm, self.lm_head = m.tok_embed, m.final_norm, m.lm_head
        self.w = {k: np.asarray(v, np.float32) for k, v in w.items()}


def block(head: MtpHead, z: np.ndarray, positions: np.ndarray,
          cache: Optional[Tuple[np.ndarray, np.ndarray]] = None, first_pos: Optional[int] = None):
    """B applied to rows z [n, h] at absolute ``positions`` (consecutive),
    attending causally to ``cache`` (keys / values of the earlier rows of the
    same depth, the first at ``first_pos``) and to earlier rows of this call.
    Returns (output [n, h], extended cache)."""
    cfg, w = head.cfg, head.w
    hq, hk, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    positions = np.asarray(positions)
    n = z.shape[0]
    u = rms_norm(z, w["attn_norm"], cfg.rms_eps)
    qkv = (u @ w["w_qkv"].T).astype(np.float32)
    q = rope(qkv[:, : hq * d].reshape(n, hq, d), positions, cfg.rope_theta)
    k = rope(qkv[:, hq * d:(hq + hk) * d].reshape(n, hk, d), positions, cfg.rope_theta)
    v = qkv[:, (hq + hk) * d:].reshape(n, hk, d)
    if cache is None:
        cache = (np.zeros((0, hk, d), np.float32), np.zeros((0, hk, d), np.float32))
        first_pos = int(positions[0])
    if cfg.wdtype != 0:       # the block's cache is held in the model's storage type, like the decoder's
        k, v = round_bf16(k), round_bf16(v)
    kk = np.concatenate([cache[0], k])
    vv = np.concatenate([cache[1], v])
    o = attention_rows(q, kk, vv, positions - first_pos, hk)     # key j sits at first_pos + j
    x = z + (o.reshape(n, hq * d) @ w["w_o"].T).astype(np.float32)
    u = rms_norm(x, w["ffn_norm"], cfg.rms_eps)
    x = x + ((_silu(u @ w["w_gate"].T) * (u @ w["w_up"].T)) @ w["w_down"].T).astype(np.float32)
    return x.astype(np.float32), (kk, vv)


def block_input(head: MtpHead, next_tokens: Sequence[int], a: np.ndarray) -> np.ndarray:
    """z = P([N_e(E(x_(p+1))); N_h(a)]) for rows given their next tokens and states a."""
    cfg, w = head.cfg, head.w
    e = head.tok_embed[np.asarray(next_tokens, np.int64)]
    cat = np.concatenate([rms_norm(e, w["enorm"], cfg.rms_eps), rms_norm(a, w["hnorm"], cfg.rms_eps)], axis=-1)
    return (cat @ w["eh_proj"].T).astype(np.float32)


def grid(head: MtpHead, b: np.ndarray, tokens: Sequence[int], p0: int, K: int) -> List[Dict[int, np.ndarray]]:
    """u_p^(k) for k = 1..K by the definition, each depth one causal pass over
    its rows (no cache reuse). b: [N, h] decoder states of rows 0..N-1;
    tokens: x_0..x_(M-1). Depth k covers rows p0 + k - 1 .. min(N + k - 2, M - 2)
    (depth 1 needs b_p; every row needs x_(p+1)). Returns one {row: u} per depth."""
    N, M = b.shape[0], len(tokens)
    out: List[Dict[int, np.ndarray]] = []
    for k in range(1, K + 1):
        lo, hi = p0 + k - 1, min(N + k - 2, M - 2)
        rows = np.arange(lo, hi + 1)
        if len(rows) == 0:
            out.append({})
            continue
        a = b[rows] if k == 1 else np.stack([out[k - 2][int(r) - 1] for r in rows])
        z = block_input(head, [tokens[int(r) + 1] for r in rows], a)
        y, _ = block(head, z, rows)
        u = rms_norm(y, head.final_norm, head.cfg.rms_eps)
        out.append({int(r): u[i] for i, r in enumerate(rows)})
    return out


def draft(head: MtpHead, b: np.ndarray, tokens: Sequence[int], p0: int, K: int) -> List[int]:
    """Drafts d_1..d_K after the committed tokens (len(tokens) == len(b) + 1:
    x_(p+1) is the last committed token, p = len(b) - 1)."""
    p = b.shape[0] - 1
    assert len(tokens) == p + 2
    ext = [int(t) for t in tokens]
    d: List[int] = []
    for k in range(1, K + 1):
        u = grid(head, b, ext, p0, k)[k - 1][p + k - 1]
        t = int(np.argmax((head.lm_head @ u).astype(np.float32)))   # first maximum: lowest index
        d.append(t)
        ext.append(t)
    return d


def spec_decode(m: OracleModel, head: MtpHead, prompt, n_new: int, K: int):
    """Speculative decoding with the draft head's own drafts and greedy
    verification: after each verify step the committed rows' states extend
    b, the head drafts K tokens after the last committed token, and the
    target keeps the longest agreeing prefix plus its own next token.
    Returns (tokens, per-step accepted counts). Visual positions carry no
    token id (the grid never reads them), so they hold 0 here."""
    cache = KVCache(m.cfg)
    x = prompt_embeddings(m, prompt)
    tr = {}
    lg = forward(m, cache, x, np.arange(len(x)), tr)
    b = tr["hidden"]
    n_vis = len(prompt.visual)
    p0 = max(n_vis - 1, 0)
    tokens = [0] * n_vis + [int(t) for t in prompt.tokens]
    out = [int(argmax_lowest(lg[-1:])[0])]
    tokens.append(out[-1])
    accepted = []
    while len(out) < n_new:
        k = min(K, n_new - len(out) - 1)
        d = draft(head, b, tokens, p0, k) if k > 0 else []
        tr = {}
        base = cache.length
        g = argmax_lowest(verify_rows(m, cache, out[-1], d, tr))
        a, bonus = accept(d, g)
        cache.truncate(base + a + 1)
        b = np.concatenate([b, tr["hidden"][: a + 1]])
        out += [int(t) for t in d[:a]] + [bonus]
        tokens += [int(t) for t in d[:a]] + [bonus]
        accepted.append(a)
    return np.array(out[:n_new], np.int32), accepted
