"""Object wrapper over the C ABI: one model handle plus convenience calls.

Device memory for visual-embedding rows and step buffers comes from PyTorch;
every computation runs in libspec.so. ``cfg`` may be any object with the
decoder shape attributes (n_layers, hidden, n_q_heads, n_kv_heads, head_dim,
n_experts, top_k, n_shared, inter, vocab, wdtype, rope_theta, rms_eps).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import binding as B


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 values that are already bf16-exact -> their bf16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    if np.any(b & 0xFFFF):
        raise ValueError("values stored as bf16 must be bf16-exact")
    return (b >> 16).astype(np.uint16)


class SpecModel:
    def __init__(self, cfg, tensors: Sequence[np.ndarray], *, page_size: int = 16, n_pages: int = 1024,
                 max_seqs: int = 1, max_ctx: int = 2048, max_draft: int = 3, max_batch: Optional[int] = None,
                 prefill_chunk: int = 0, stream=None):
        import torch
        self.torch = torch
        self.cfg = cfg
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.c = B.make_config(
            n_layers=cfg.n_layers, hidden=cfg.hidden, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
            head_dim=cfg.head_dim, n_experts=cfg.n_experts, top_k=cfg.top_k, n_shared=cfg.n_shared,
            inter=cfg.inter, vocab=cfg.vocab, wdtype=cfg.wdtype, page_size=page_size, n_pages=n_pages,
            max_seqs=max_seqs, max_ctx=max_ctx, max_draft=max_draft,
            max_batch=max_batch if max_batch is not None else max_seqs, prefill_chunk=prefill_chunk,
            rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps)
        self.K = max_draft
        self.h = B.spec_init_model(self.c, tensors, int(self.stream.cuda_stream))
        self._tied = list(tensors[:3])     # embedding, final norm, LM head: shared with a draft head

    # -- FastMTP draft head ----------------------------------------------------
    MTP_ORDER = ("enorm", "hnorm", "eh_proj", "attn_norm", "w_qkv", "w_o", "ffn_norm", "w_gate", "w_up", "w_down")

    def attach_mtp(self, weights: dict, inter: int) -> None:
        """Attach a draft head: ``weights`` maps the head's tensor names to
        float32 arrays (bf16-exact matrices for bf16 / e4m3 decoders)."""
        enc = []
        for name in self.MTP_ORDER:
            a = np.ascontiguousarray(weights[name], np.float32)
            if not name.endswith("norm") and self.cfg.wdtype != B.SPEC_F32:
                a = bf16_bits(a)
            enc.append(a)
        B.spec_mtp_init(self.h, self._tied + enc, inter)

    def mtp_draft(self, seq: int, K: int) -> list:
        return [int(t) for t in B.spec_mtp_draft(self.h, seq, K)]

    def mtp_debug_draft(self, seq: int, K: int, states_cap: int = 512):
        """(drafts, fp32 logits [K, vocab] of each depth's draft row, the
        decoder's final residual rows [n, hidden] the call read for depth 1)."""
        torch = self.torch
        out = torch.empty((K, self.cfg.vocab), dtype=torch.float32, device="cuda")
        st = self._ready(torch.empty((states_cap, self.cfg.hidden), dtype=torch.float32, device="cuda"))
        d, n = B.spec_mtp_debug_draft(self.h, seq, K, out, st, states_cap)
        self.stream.synchronize()
        return [int(t) for t in d], out.cpu().numpy(), st[:n].cpu().numpy()

    def close(self) -> None:
        if self.h:
            B.spec_free_model(self.h)
            self.h = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- prompts ---------------------------------------------------------------
    def visual_to_device(self, visual: np.ndarray):
        torch = self.torch
        if len(visual) == 0:
            return None
        if self.cfg.wdtype == B.SPEC_F32:
            return torch.from_numpy(np.ascontiguousarray(visual, np.float32)).cuda()
        return torch.from_numpy(bf16_bits(visual).view(np.int16)).cuda()

    def _ready(self, t):
        # uploads run on torch's current stream; the library uses its own
        self.torch.cuda.current_stream().synchronize()
        return t

    def prefill(self, seq: int, visual: np.ndarray, tokens, prefix_id: int = -1) -> int:
        dev = self._ready(self.visual_to_device(visual))
        return B.spec_prefill(self.h, seq, prefix_id, dev, len(visual), tokens)

    def register_prefix(self, tokens) -> int:
        return B.spec_register_prefix(self.h, tokens)

    # -- steps -----------------------------------------------------------------
    def verify(self, seq: int, drafts) -> tuple:
        return B.spec_verify_step(self.h, seq, drafts)

    def verify_batch(self, seq_ids, drafts: np.ndarray, n_draft) -> tuple:
        return B.spec_verify_step_batch(self.h, seq_ids, np.asarray(drafts, np.int32).reshape(-1), n_draft)

    def verify_sample_batch(self, seq_ids, drafts: np.ndarray, n_draft, u_accept: np.ndarray,
                            u_sample: np.ndarray, temperature: float) -> tuple:
        """Rejection-sampling verify step (spec_verify_step_sample_batch):
        (accepted, appended token) per sequence."""
        return B.spec_verify_step_sample_batch(self.h, seq_ids, np.asarray(drafts, np.int32).reshape(-1), n_draft,
                                               u_accept, u_sample, temperature)

    def debug_logits(self, seq_ids, drafts: np.ndarray) -> np.ndarray:
        torch = self.torch
        n = len(seq_ids) * (self.K + 1)
        out = self._ready(torch.empty((n, self.cfg.vocab), dtype=torch.float32, device="cuda"))
        B.spec_debug_logits(self.h, seq_ids, np.asarray(drafts, np.int32).reshape(-1), out)
        self.stream.synchronize()
        return out.cpu().numpy()

    def tokens(self, seq: int) -> np.ndarray:
        return B.spec_seq_tokens(self.h, seq)

    def length(self, seq: int) -> int:
        return B.spec_seq_info(self.h, seq)[0]

    def block_table(self, seq: int) -> np.ndarray:
        return B.spec_seq_block_table(self.h, seq)

    def release(self, seq: int) -> None:
        B.spec_release_seq(self.h, seq)
