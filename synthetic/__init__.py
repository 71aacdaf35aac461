"""Seeded synthetic inputs for the speculative-decoding verify step.

This module is shared by the CPU oracle (``oracle/``), the tests and the
benchmark. It holds no arithmetic of the method itself: it only draws and
encodes *inputs* -- model weights, visual-embedding rows, prompt token ids,
output lengths and the synthetic drafter's proposals. Everything the verify
step computes from those inputs lives elsewhere (the oracle on the CPU, the
CUDA library on the GPU), and the two never share code.

Encodings produced here (the byte formats the C-ABI consumes):

* ``f32``  -- IEEE binary32, little endian.
* ``bf16`` -- the upper 16 bits of binary32 after round-to-nearest-even.
* ``e4m3`` -- OCP FP8 E4M3 ("fn" variant: no infinities, S.1111.111 = NaN,
  largest finite 448), round-to-nearest-even with saturation to +-448, plus one
  fp32 scale per output channel (row): ``s_o = max_j |W_oj| / 448`` and
  ``code_oj = e4m3(W_oj / s_o)``.
* ``nvfp4`` -- 4-bit E2M1 codes with one E4M3 scale per 16 consecutive
  elements of a row and one fp32 scale per matrix (per expert for stacked
  experts), ``value = e2m1 * e4m3(block scale) * tensor scale``
  (``quantize_nvfp4``). A [rows, K] matrix is stored as its codes packed two
  per byte -- element 2j in the low nibble of byte j of the row, element 2j+1
  in the high nibble -- rows * K / 2 bytes, followed by the block scale codes
  [rows, K / 16]; stacked experts store one such record per expert. The
  tensor scales go in the matrix's scale tensor (fp32, one per matrix).

Model shapes and workload recipes follow the five workloads the pages
describe for document-OCR serving (Jina-OCR-v1, section 3 "model
architecture" and the jina-ocr-v1 release article; the OCRia-1 report guide,
"inference stack"): a DeepSeekMoE-style 3B decoder with 64 routed + 2 shared
experts (top-6), 256 + 100 n visual tokens per page, about 1,085 output tokens
per page, K = 3 drafts (FastMTP) or a 31-token block draft (DFlash2).
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

F32, BF16, FP8, NVFP4 = 0, 1, 2, 3    # storage dtype codes (same numbering as the C-ABI)
DTYPE_NAMES = {F32: "f32", BF16: "bf16", FP8: "e4m3", NVFP4: "nvfp4"}

# --------------------------------------------------------------------------- #
# Model configuration
# --------------------------------------------------------------------------- #


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Decoder shape. ``n_experts == 0`` means a dense SwiGLU FFN, which is
    represented as one always-on ("shared") expert of width ``inter``."""
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    n_shared: int
    inter: int
    vocab: int
    wdtype: int = F32
    rope_theta: float = 10000.0
    rms_eps: float = 1e-6
    init_std: float = 0.02

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def n_ffn(self) -> int:          # routed + shared experts stored together
        return self.n_experts + self.n_shared

    def active_params(self) -> int:
        """Parameters touched by one token (decoder + LM head, no embedding)."""
        h, d = self.hidden, self.head_dim
        attn = self.qkv_rows * h + h * self.n_q_heads * d
        expert = 3 * self.inter * h
        ffn = (self.top_k + self.n_shared) * expert + self.n_experts * h
        return self.n_layers * (attn + ffn) + self.vocab * h


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic serving workload (model + prompts + drafter + lengths)."""
    name: str
    model: ModelConfig
    batch: int                    # concurrent sequences
    n_draft: int                  # K drafts per verify step
    drafter: str                  # "iid" (per-position match prob q) or "geometric"
    q: float                      # iid match prob, or geometric stop prob p
    visual: Tuple[int, ...]       # (base, step, n_max): base + step * n, n ~ U{0..n_max}
    n_text: int                   # instruction token ids after the visual rows
    shared_prefix: int            # token ids of a prefix shared by every sequence
    out_len: Tuple[float, ...]    # (fixed,) or (mean, std, lo, hi) clipped normal
    page_size: int = 16


TINY = ModelConfig("tiny-fp32-moe", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=4,
                   head_dim=64, n_experts=8, top_k=2, n_shared=1, inter=128, vocab=1024,
                   wdtype=F32)
MOE3B = ModelConfig("deepseek-3b-moe-shape", n_layers=12, hidden=1280, n_q_heads=10,
                    n_kv_heads=10, head_dim=128, n_experts=64, top_k=6, n_shared=2,
                    inter=896, vocab=129280, wdtype=BF16)
MOE3B_FP8 = dataclasses.replace(MOE3B, name="deepseek-3b-moe-shape-fp8", wdtype=FP8)
MOE3B_NVFP4 = dataclasses.replace(MOE3B, name="deepseek-3b-moe-shape-nvfp4", wdtype=NVFP4)
DENSE4B = ModelConfig("qwen3-4b-shape", n_layers=36, hidden=2560, n_q_heads=32,
                      n_kv_heads=8, head_dim=128, n_experts=0, top_k=0, n_shared=1,
                      inter=9728, vocab=151936, wdtype=BF16, rope_theta=1_000_000.0)

WORKLOADS: Dict[str, Workload] = {
    # tiny fp32 MoE, batch 1: 64 visual + 8 ids, K=3 with match prob 0.6, 128 tokens
    "tiny_fp32_b1": Workload("tiny_fp32_b1", TINY, batch=1, n_draft=3, drafter="iid", q=0.6,
                             visual=(64, 0, 0), n_text=8, shared_prefix=0, out_len=(128,)),
    # 3B-MoE bf16, batch 1: 256 visual + 16 ids, K=3 q=0.576, 1,085 tokens
    "moe3b_bf16_b1": Workload("moe3b_bf16_b1", MOE3B, batch=1, n_draft=3, drafter="iid",
                              q=0.576, visual=(256, 0, 0), n_text=16, shared_prefix=0,
                              out_len=(1085,)),
    # 3B-MoE bf16 at concurrency 32: 256 + 100 n visual, N(1085, 300^2) in [200, 4000]
    "moe3b_bf16_c32": Workload("moe3b_bf16_c32", MOE3B, batch=32, n_draft=3, drafter="iid",
                               q=0.576, visual=(256, 100, 9), n_text=16, shared_prefix=0,
                               out_len=(1085.0, 300.0, 200, 4000)),
    # dense Qwen3-4B shape, 31-token block draft, geometric accepted prefix p=0.15
    "dense4b_bf16_b1": Workload("dense4b_bf16_b1", DENSE4B, batch=1, n_draft=31,
                                drafter="geometric", q=0.15, visual=(1288, 0, 0), n_text=0,
                                shared_prefix=0, out_len=(1200,)),
    "dense4b_bf16_b8": Workload("dense4b_bf16_b8", DENSE4B, batch=8, n_draft=31,
                                drafter="geometric", q=0.15, visual=(1288, 0, 0), n_text=0,
                                shared_prefix=0, out_len=(1200,)),
    # the batch-1 3B-MoE workload with NVFP4 attention and expert weights
    "moe3b_nvfp4_b1": Workload("moe3b_nvfp4_b1", MOE3B_NVFP4, batch=1, n_draft=3, drafter="iid",
                               q=0.576, visual=(256, 0, 0), n_text=16, shared_prefix=0,
                               out_len=(1085,)),
    # 3B-MoE with e4m3 weights at concurrency 64, shared 64-token prefix
    "moe3b_fp8_c64": Workload("moe3b_fp8_c64", MOE3B_FP8, batch=64, n_draft=3, drafter="iid",
                              q=0.576, visual=(256, 100, 9), n_text=0, shared_prefix=64,
                              out_len=(1085.0, 300.0, 200, 4000)),
}


def scaled(model: ModelConfig, **kw) -> ModelConfig:
    """A smaller model of the same family (tests use these)."""
    return dataclasses.replace(model, **kw)


# --------------------------------------------------------------------------- #
# Tensor list (the order the C-ABI documents for spec_init_model)
# --------------------------------------------------------------------------- #
PER_LAYER = ("attn_norm", "w_qkv", "s_qkv", "w_o", "s_o", "ffn_norm", "w_router",
             "w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")
N_GLOBAL = 3  # tok_embed, final_norm, lm_head


def tensor_specs(cfg: ModelConfig) -> List[Tuple[str, Tuple[int, ...], int, int]]:
    """(name, shape, storage dtype, layer) for every tensor, in C-ABI order.

    Storage: norms and scales are always f32; the router, embedding and LM
    head are f32 for f32 models and bf16 otherwise; attention and expert
    matrices use ``cfg.wdtype`` (their shape is the logical [.., rows, K]; an
    nvfp4 array holds the packed record, ``nvfp4_bytes`` per matrix). Scales:
    one per output row for e4m3, one per matrix for nvfp4. Absent tensors
    (scales of other models, the router of a dense model) have shape (0,)."""
    h, d = cfg.hidden, cfg.head_dim
    side = F32 if cfg.wdtype == F32 else BF16
    fp8 = cfg.wdtype == FP8
    q4 = cfg.wdtype == NVFP4
    F = cfg.n_ffn

    def sc(fp8_shape, q4_shape):
        return fp8_shape if fp8 else q4_shape if q4 else (0,)
    out = [("tok_embed", (cfg.vocab, h), side, -1),
           ("final_norm", (h,), F32, -1),
           ("lm_head", (cfg.vocab, h), side, -1)]
    for l in range(cfg.n_layers):
        out += [
            ("attn_norm", (h,), F32, l),
            ("w_qkv", (cfg.qkv_rows, h), cfg.wdtype, l),
            ("s_qkv", sc((cfg.qkv_rows,), (1,)), F32, l),
            ("w_o", (h, cfg.n_q_heads * d), cfg.wdtype, l),
            ("s_o", sc((h,), (1,)), F32, l),
            ("ffn_norm", (h,), F32, l),
            ("w_router", (cfg.n_experts, h) if cfg.n_experts else (0,), side, l),
            ("w_gate", (F, cfg.inter, h), cfg.wdtype, l),
            ("s_gate", sc((F, cfg.inter), (F,)), F32, l),
            ("w_up", (F, cfg.inter, h), cfg.wdtype, l),
            ("s_up", sc((F, cfg.inter), (F,)), F32, l),
            ("w_down", (F, h, cfg.inter), cfg.wdtype, l),
            ("s_down", sc((F, h), (F,)), F32, l),
        ]
    return out


# --------------------------------------------------------------------------- #
# Encodings
# --------------------------------------------------------------------------- #

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
            >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_positive_table() -> np.ndarray:
    """Values of the 127 non-negative finite E4M3 codes 0x00..0x7E."""
    vals = np.empty(127, dtype=np.float64)
    for c in range(127):
        e, m = c >> 3, c & 7
        vals[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3_POS = _e4m3_positive_table()


def f32_to_e4m3(a: np.ndarray) -> np.ndarray:
    """binary32 -> E4M3 codes, round to nearest (ties to even code), saturating."""
    a = np.asarray(a, dtype=np.float32)
    mag = np.minimum(np.abs(a).astype(np.float64), 448.0)
    hi = np.searchsorted(_E4M3_POS, mag, side="left").clip(0, 126)   # first >= mag
    lo = np.maximum(hi - 1, 0)
    dlo = mag - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(mag == _E4M3_POS[hi], hi.astype(np.uint8), code)
    sign = (np.signbit(a) & (code != 0)).astype(np.uint8) << np.uint8(7)
    return (code | sign).astype(np.uint8)


def quantize_rows_e4m3(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-output-channel (last axis reduced) e4m3 quantisation -> (codes, scales)."""
    amax = np.max(np.abs(w), axis=-1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = f32_to_e4m3(w / scale[..., None])
    return codes, scale


_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f32_to_e2m1(a: np.ndarray) -> np.ndarray:
    """binary32 -> FP4 E2M1 codes (one per byte, low nibble), round to nearest
    (ties to the even code), saturating at +-6; -0 encodes as 0."""
    a = np.asarray(a, dtype=np.float32)
    mag = np.minimum(np.abs(a).astype(np.float64), 6.0)
    hi = np.searchsorted(_E2M1_POS, mag, side="left").clip(0, 7)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = mag - _E2M1_POS[lo], _E2M1_POS[hi] - mag
    code = np.where((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)), hi, lo)
    code = np.where(mag == _E2M1_POS[hi], hi, code).astype(np.uint8)
    return (code | ((np.signbit(a) & (code != 0)).astype(np.uint8) << np.uint8(3))).astype(np.uint8)


def nvfp4_bytes(rows: int, K: int) -> int:
    """Bytes of one packed nvfp4 matrix record: codes, then block scales."""
    return rows * K // 2 + rows * K // 16


def pack_nvfp4(codes: np.ndarray, block_scales: np.ndarray) -> np.ndarray:
    """One matrix record: codes [rows, K] two per byte (element 2j in the low
    nibble of byte j), then the block scale codes [rows, K/16]; flat uint8."""
    c = np.asarray(codes, dtype=np.uint8)
    packed = (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)
    return np.concatenate([packed.reshape(-1), np.asarray(block_scales, dtype=np.uint8).reshape(-1)])


def quantize_nvfp4(w: np.ndarray):
    """NVFP4 encoding of w [..., K] (K a multiple of 16): tensor scale
    amax(w) / (6 * 448); per 16-element block an E4M3 scale of
    amax(block) / (6 * tensor scale); codes E2M1(w / (block scale * tensor
    scale)). Returns (codes [..., K], block scale codes [..., K/16], tensor scale)."""
    w = np.asarray(w, dtype=np.float32)
    amax = float(np.max(np.abs(w)))
    ts = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blocks = w.reshape(*w.shape[:-1], -1, 16)
    bs_codes = f32_to_e4m3(np.max(np.abs(blocks), axis=-1) / (6.0 * ts))
    bs = _E4M3_POS[bs_codes & 0x7F].astype(np.float64)
    denom = np.where(bs > 0, bs * float(ts), 1.0)[..., None]
    codes = f32_to_e2m1((blocks / denom).astype(np.float32)).reshape(w.shape)
    return codes, bs_codes, float(ts)


# --------------------------------------------------------------------------- #
# Weights
# --------------------------------------------------------------------------- #

def _normal(seed: int, tensor_index: int, sub: int, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64([seed, tensor_index, sub]))
    out = g.standard_normal(int(np.prod(shape)), dtype=np.float32)
    out *= np.float32(std)
    return out.reshape(shape)


@dataclasses.dataclass
class Weights:
    """Encoded weight tensors in C-ABI order (``arrays[i]`` is f32, uint16 bf16
    bits or uint8 e4m3 codes, per ``specs[i][2]``)."""
    cfg: ModelConfig
    specs: List[Tuple[str, Tuple[int, ...], int, int]]
    arrays: List[np.ndarray]

    def get(self, name: str, layer: int = -1) -> np.ndarray:
        for (n, _, _, l), a in zip(self.specs, self.arrays):
            if n == name and l == layer:
                return a
        raise KeyError((name, layer))

    @property
    def nbytes(self) -> int:
        return sum(a.nbytes for a in self.arrays)


def generate_weights(cfg: ModelConfig, seed: int = 0, threads: Optional[int] = None,
                     norm_gamma_std: float = 0.0) -> Weights:
    """Draw every matrix ~ N(0, init_std^2) from a per-(tensor, expert) PCG64
    stream keyed by ``seed``; norms are ones (or 1 + N(0, norm_gamma_std^2) when a
    test asks for non-trivial gains). Matrices are then encoded in the storage
    dtype. Generation is deterministic and independent of ``threads``."""
    specs = tensor_specs(cfg)
    arrays: List[Optional[np.ndarray]] = [None] * len(specs)
    threads = threads or min(32, os.cpu_count() or 1)

    # scale tensors are filled when their matrix is quantised
    scale_of = {"w_qkv": "s_qkv", "w_o": "s_o", "w_gate": "s_gate", "w_up": "s_up",
                "w_down": "s_down"}
    index = {(n, l): i for i, (n, _, _, l) in enumerate(specs)}

    def encode(mat: np.ndarray, dtype: int):
        if dtype == F32:
            return mat, None
        if dtype == BF16:
            return f32_to_bf16_bits(mat), None
        if dtype == NVFP4:
            codes, bs, ts = quantize_nvfp4(mat)
            return pack_nvfp4(codes, bs), np.float32(ts)
        return quantize_rows_e4m3(mat)

    jobs = []
    for i, (name, shape, dtype, layer) in enumerate(specs):
        if name.startswith("s_") or int(np.prod(shape)) == 0:
            continue
        jobs.append(i)

    def run(i: int):
        name, shape, dtype, layer = specs[i]
        if name.endswith("norm"):
            if norm_gamma_std > 0:
                g = 1.0 + _normal(seed, i, 0, shape, norm_gamma_std)
            else:
                g = np.ones(shape, dtype=np.float32)
            arrays[i] = g.astype(np.float32)
            return
        if len(shape) == 3:   # stacked experts: one stream per expert
            parts, scales = [], []
            for e in range(shape[0]):
                enc, sc = encode(_normal(seed, i, e + 1, shape[1:], cfg.init_std), dtype)
                parts.append(enc)
                scales.append(sc)
            arrays[i] = np.stack(parts)
            if dtype in (FP8, NVFP4):
                arrays[index[(scale_of[name], layer)]] = np.stack(scales).astype(np.float32)
        else:
            enc, sc = encode(_normal(seed, i, 0, shape, cfg.init_std), dtype)
            arrays[i] = enc
            if sc is not None:
                arrays[index[(scale_of[name], layer)]] = np.atleast_1d(np.asarray(sc, np.float32))

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(run, jobs))
    for i, (name, shape, dtype, layer) in enumerate(specs):
        if arrays[i] is None:
            npdt = {F32: np.float32, BF16: np.uint16, FP8: np.uint8, NVFP4: np.uint8}[dtype]
            arrays[i] = np.zeros(shape, dtype=npdt)
    return Weights(cfg, specs, arrays)  # type: ignore[arg-type]


# --------------------------------------------------------------------------- #
# Draft head (FastMTP) weights
# --------------------------------------------------------------------------- #
MTP_TENSORS = ("enorm", "hnorm", "eh_proj", "attn_norm", "w_qkv", "w_o", "ffn_norm", "w_gate", "w_up", "w_down")


def mtp_inter(cfg: ModelConfig) -> int:
    """Width of the draft block's dense SwiGLU: the FFN width one token meets
    in the decoder ((top_k + n_shared) * inter; inter for a dense decoder)."""
    return (cfg.top_k + cfg.n_shared) * cfg.inter if cfg.n_experts else cfg.inter


def mtp_tensor_shapes(cfg: ModelConfig) -> Dict[str, Tuple[int, ...]]:
    h, d, f = cfg.hidden, cfg.head_dim, mtp_inter(cfg)
    return {"enorm": (h,), "hnorm": (h,), "eh_proj": (h, 2 * h), "attn_norm": (h,),
            "w_qkv": (cfg.qkv_rows, h), "w_o": (h, cfg.n_q_heads * d), "ffn_norm": (h,),
            "w_gate": (f, h), "w_up": (f, h), "w_down": (h, f)}


def generate_mtp_weights(cfg: ModelConfig, seed: int = 0, norm_gamma_std: float = 0.0) -> Dict[str, np.ndarray]:
    """The draft head's own tensors (the embedding, output norm and LM head are
    the decoder's), float32: matrices ~ N(0, init_std^2) from PCG64 streams
    keyed by (seed, 10,000 + tensor index) -- disjoint from the decoder's --
    rounded to bf16 values for bf16 / fp8 models (the head stays bf16); norm
    gains ones, or 1 + N(0, norm_gamma_std^2)."""
    out = {}
    for i, (name, shape) in enumerate(mtp_tensor_shapes(cfg).items()):
        if name.endswith("norm"):
            g = 1.0 + _normal(seed, 10_000 + i, 0, shape, norm_gamma_std) if norm_gamma_std > 0 else np.ones(shape)
            out[name] = np.asarray(g, np.float32)
            continue
        m = _normal(seed, 10_000 + i, 0, shape, cfg.init_std)
        out[name] = m if cfg.wdtype == F32 else bf16_bits_to_f32(f32_to_bf16_bits(m))
    return out


# --------------------------------------------------------------------------- #
# Prompts, output lengths
# --------------------------------------------------------------------------- #

@dataclasses.dataclass
class Prompt:
    """One sequence's prompt: ``prefix_tokens`` (shared across sequences, may be
    empty) ++ ``visual`` rows ++ ``tokens``. ``visual`` is f32 [n_vis, hidden]
    holding values exactly representable in the model's activation dtype."""
    prefix_tokens: np.ndarray
    visual: np.ndarray
    tokens: np.ndarray
    out_len: int

    @property
    def length(self) -> int:
        return len(self.prefix_tokens) + len(self.visual) + len(self.tokens)


def make_prompts(w: Workload, n_seq: Optional[int] = None, seed: int = 1,
                 length_seed: int = 3) -> List[Prompt]:
    """Seeded synthetic prompts for ``n_seq`` sequences of workload ``w``.

    Visual rows ~ N(0, 1) (rounded to bf16 for bf16/fp8 models so both sides
    see identical inputs); token ids ~ U[0, vocab); the visual count is
    base + step * n with n ~ U{0..n_max}; output lengths are fixed or a normal
    clipped to [lo, hi] and rounded to an integer."""
    cfg = w.model
    n_seq = n_seq if n_seq is not None else w.batch
    gp = np.random.Generator(np.random.PCG64([seed, 0xC0FFEE]))
    prefix = gp.integers(0, cfg.vocab, size=w.shared_prefix, dtype=np.int64).astype(np.int32)
    gl = np.random.Generator(np.random.PCG64([length_seed, 0x1E]))
    out = []
    for s in range(n_seq):
        g = np.random.Generator(np.random.PCG64([seed, s]))
        base, step, nmax = w.visual
        n_vis = base + step * int(g.integers(0, nmax + 1)) if step else base
        vis = g.standard_normal((n_vis, cfg.hidden), dtype=np.float32)
        if cfg.wdtype != F32:
            vis = bf16_bits_to_f32(f32_to_bf16_bits(vis))
        toks = g.integers(0, cfg.vocab, size=w.n_text, dtype=np.int64).astype(np.int32)
        if len(w.out_len) == 1:
            n_out = int(w.out_len[0])
        else:
            mu, sd, lo, hi = w.out_len
            n_out = int(np.clip(round(gl.normal(mu, sd)), lo, hi))
        out.append(Prompt(prefix.copy(), vis, toks, n_out))
    return out


# --------------------------------------------------------------------------- #
# Synthetic drafter
# --------------------------------------------------------------------------- #

class Drafter:
    """Seeded synthetic drafter standing in for FastMTP / DFlash2 proposals.

    Given the reference greedy continuation ``ref`` of a sequence (``ref[i]`` is
    the i-th generated token) and the number of tokens committed so far ``n``,
    it proposes ``k`` drafts meant to continue after ``ref[n-1]``:

    * ``iid``: draft j equals ``ref[n - 1 + j]`` with probability ``q``,
      otherwise a token uniform over the other ``vocab - 1`` ids;
    * ``geometric``: an intended accepted length L ~ P(L = l) = (1-p)^l p,
      capped at k; drafts 1..L are reference tokens, draft L+1 is a wrong
      token, the rest are uniform over the vocabulary.

    Draws come from a PCG64 stream keyed by (seed, sequence id, step index), so
    the proposals are reproducible whatever the batch composition."""

    def __init__(self, mode: str, q: float, vocab: int, seed: int = 2):
        assert mode in ("iid", "geometric")
        self.mode, self.q, self.vocab, self.seed = mode, q, vocab, seed

    def _wrong(self, g: np.random.Generator, ref: int) -> int:
        r = int(g.integers(0, self.vocab - 1))
        return r + 1 if r >= ref else r

    def propose(self, ref: Sequence[int], n: int, k: int, seq: int, step: int) -> np.ndarray:
        g = np.random.Generator(np.random.PCG64([self.seed, seq, step]))
        out = np.empty(k, dtype=np.int32)
        if self.mode == "iid":
            hits = g.random(k) < self.q
            for j in range(k):
                i = n - 1 + (j + 1)
                r = int(ref[i]) if i < len(ref) else -1
                if r >= 0 and hits[j]:
                    out[j] = r
                else:
                    out[j] = self._wrong(g, max(r, 0)) if r >= 0 else int(g.integers(0, self.vocab))
        else:
            p = self.q
            L = 0
            while L < k and g.random() >= p:
                L += 1
            for j in range(k):
                i = n - 1 + (j + 1)
                r = int(ref[i]) if i < len(ref) else -1
                if j < L and r >= 0:
                    out[j] = r
                elif j == L and r >= 0:
                    out[j] = self._wrong(g, r)
                else:
                    out[j] = int(g.integers(0, self.vocab))
        return out


def expected_accept_iid(q: float, k: int) -> float:
    """E[accepted drafts] when each draft matches independently with prob q."""
    return sum(q ** i for i in range(1, k + 1))


def expected_accept_geometric(p: float, k: int) -> float:
    """E[min(L, k)] for P(L = l) = (1-p)^l p."""
    return sum((1 - p) ** i for i in range(1, k + 1))


def draft_schedule(drafter: Drafter, ref: Sequence[int], n_steps: int, k: int, seq: int = 0):
    """Plan a drafter's proposals for ``n_steps`` consecutive verify steps of one
    sequence whose greedy continuation is ``ref`` (ref[0] = first generated
    token). Because the synthetic drafter is built around the reference, it
    knows how many of its proposals agree with it: step s proposes from the
    committed count n_s, and n_(s+1) = n_s + (leading agreeing drafts) + 1.
    Returns (drafts [n_steps, k] int32, agreeing prefix lengths [n_steps],
    committed counts before each step [n_steps])."""
    drafts = np.zeros((n_steps, k), np.int32)
    agree = np.zeros(n_steps, np.int32)
    n_before = np.zeros(n_steps, np.int64)
    n = 1
    for s in range(n_steps):
        d = drafter.propose(ref, n, k, seq, s)
        drafts[s] = d
        a = 0
        while a < k and n + a < len(ref) and int(d[a]) == int(ref[n + a]):
            a += 1
        agree[s] = a
        n_before[s] = n
        n += a + 1
    return drafts, agree, n_before
