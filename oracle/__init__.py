"""CPU oracle for the greedy, lossless speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product (the CUDA library and its Python binding) never imports,
links or calls anything here, and nothing here imports the product.

What it computes is the plain definition the speculative method reaches
exactly: ordinary token-by-token greedy decoding of a random-init decoder
(Jina-OCR-v1 abstract: greedy verification makes decoding lossless; the
jina-ocr-v1 release article: output identical to autoregressive greedy
decoding; the end-to-end OCR explainer, section 6.1 "draft-verify" and
section 7, the speculative loop). Everything is numpy float32 (the precision
the method's description fixes for its checker), with library matmuls as the
only primitives and no blocking, fusion or reordering beyond the definitions.

Readings of points the pages leave open (each one mirrored, not shared, by the
GPU path):

* RMSNorm(z) = z / sqrt(mean(z^2) + eps) * gamma, eps = 1e-6.
* RoPE: rotate-half pairing (i, i + d/2), angle p * theta^(-2i/d) evaluated in
  float64 and rounded to float32 cos/sin; positions are absolute from 0,
  visual rows included.
* Attention scale 1/sqrt(head_dim); GQA maps q head h to kv head
  floor(h * H_kv / H_q).
* MoE: softmax over all experts in float32, top-k ordered by (probability
  descending, expert id ascending), no renormalisation; shared experts are
  always on with weight 1; expert F(u) = W_d (silu(W_g u) * (W_u u)).
* Greedy argmax and the acceptance rule break ties toward the lowest index.
* Acceptance: a = the longest prefix of drafts with d_j = g_(j-1); the bonus
  token g_a is always committed, so a verify step commits a + 1 tokens.
* The KV cache holds keys and values in the model's activation storage type
  (bf16 for bf16 and e4m3-weight models, f32 for f32 models), as the model's
  own state; all arithmetic on them is float32.

``oracle.sampling`` holds the stochastic counterpart of the acceptance rule
(rejection-sampling verification), pinned by tests/test_oracle_sampling.py.

Parity pins (tests/test_oracle_*.py): brute-force recompute without a cache,
spec == greedy for random / all-correct / all-wrong drafts, dense special
case, one-key attention, RoPE identity and relative-position property, e4m3 and
bf16 decodes against the format definitions, and the page counts of the
workloads. Logit *values* beyond these properties are parity unpinned except
through these checks: the pages print no worked example.
"""
from .model import (OracleModel, KVCache, rms_norm, rope, attention_rows, moe_ffn,
                    forward, prompt_embeddings, greedy_decode, spec_decode, accept,
                    brute_force_logits, teacher_forced_logits, verify_rows,
                    decode_bf16, decode_e4m3, decode_e2m1, decode_nvfp4, unpack_nvfp4, route, commit_pages,
                    round_bf16)

__all__ = ["OracleModel", "KVCache", "rms_norm", "rope", "attention_rows", "moe_ffn",
           "forward", "prompt_embeddings", "greedy_decode", "spec_decode", "accept",
           "brute_force_logits", "teacher_forced_logits", "verify_rows", "decode_bf16",
           "decode_e4m3", "decode_e2m1", "decode_nvfp4", "unpack_nvfp4", "route", "commit_pages", "round_bf16"]
