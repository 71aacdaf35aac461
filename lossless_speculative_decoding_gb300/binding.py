"""ctypes binding of libspec.so (argument marshalling only).

Every function here has the name of the C entry point it calls (declared in
``include/spec.h``) and does no computation of its own: all work of the verify
step runs in the library's CUDA kernels. Loading fails loudly when the
library has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspec.so")

SPEC_F32, SPEC_BF16, SPEC_FP8, SPEC_NVFP4 = 0, 1, 2, 3
SPEC_ERR_ARG, SPEC_ERR_NO_PAGES, SPEC_ERR_CUDA, SPEC_ERR_STATE, SPEC_ERR_NOMEM, SPEC_ERR_UNSUPPORTED = -1, -2, -3, -4, -5, -6
ERRORS = {-1: "SPEC_ERR_ARG", -2: "SPEC_ERR_NO_PAGES", -3: "SPEC_ERR_CUDA", -4: "SPEC_ERR_STATE",
          -5: "SPEC_ERR_NOMEM", -6: "SPEC_ERR_UNSUPPORTED"}


class SpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class spec_kernel_stat(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_float), ("launches", ctypes.c_int32), ("units", ctypes.c_int64)]


SPEC_KCLASS_COUNT = 11


class spec_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "n_experts", "top_k", "n_shared",
        "inter", "vocab", "wdtype", "page_size", "n_pages", "max_seqs", "max_ctx", "max_draft",
        "max_batch", "prefill_chunk")] + [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


_I32P = ctypes.POINTER(ctypes.c_int32)
_lib: Optional[ctypes.CDLL] = None

# (name, restype, argtypes) of every exported entry point
_SIGS = [
    ("spec_tensor_count", ctypes.c_int, [ctypes.POINTER(spec_config)]),
    ("spec_tensor_bytes", ctypes.c_int64, [ctypes.POINTER(spec_config), ctypes.c_int]),
    ("spec_init_model", ctypes.c_int, [ctypes.POINTER(spec_config), ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)]),
    ("spec_free_model", ctypes.c_int, [ctypes.c_void_p]),
    ("spec_register_prefix", ctypes.c_int, [ctypes.c_void_p, _I32P, ctypes.c_int, _I32P]),
    ("spec_release_prefix", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("spec_prefill", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                    ctypes.c_int, _I32P, ctypes.c_int, _I32P]),
    ("spec_verify_step", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P, ctypes.c_int, _I32P, _I32P]),
    ("spec_verify_step_batch", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, _I32P, _I32P, _I32P, _I32P,
                                              _I32P]),
    ("spec_verify_step_batch_dev", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p]),
    ("spec_verify_step_sample_batch", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, _I32P, _I32P, _I32P,
                                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, _I32P,
                                                     _I32P]),
    ("spec_verify_step_sample_dev", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                                   ctypes.c_void_p]),
    ("spec_reserve_seq", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int]),
    ("spec_sync_seqs", ctypes.c_int, [ctypes.c_void_p]),
    ("spec_release_seq", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("spec_seq_info", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P, _I32P]),
    ("spec_seq_tokens", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P, ctypes.c_int]),
    ("spec_seq_block_table", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P, ctypes.c_int, _I32P]),
    ("spec_free_pages", ctypes.c_int, [ctypes.c_void_p]),
    ("spec_debug_logits", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, _I32P, _I32P, ctypes.c_void_p]),
    ("spec_step_launches", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    ("spec_mtp_init", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    ("spec_mtp_draft", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int, _I32P]),
    ("spec_mtp_debug_draft", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int, _I32P, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int, _I32P]),
    ("spec_profile_steps_dev", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                              ctypes.POINTER(spec_kernel_stat), ctypes.c_int]),
    ("spec_kernel_class_name", ctypes.c_char_p, [ctypes.c_int]),
    ("spec_io_bytes", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_int64)]),
    ("spec_lmhead_argmax_scratch_bytes", ctypes.c_int64, [ctypes.c_int, ctypes.c_int]),
    ("spec_lmhead_argmax", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t]),
    ("spec_lmhead_argmax_noalloc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                                                  ctypes.c_void_p, ctypes.c_size_t]),
    ("spec_tc_gemm_test", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]),
    ("spec_rejection_sample", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]),
    ("spec_rejection_sample_ws_bytes", ctypes.c_int64, [ctypes.c_int, ctypes.c_int]),
    ("spec_rejection_sample_ws", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_size_t, ctypes.c_size_t]),
    ("spec_strerror", ctypes.c_char_p, [ctypes.c_int]),
    ("spec_last_error", ctypes.c_char_p, []),
    ("spec_pool_create", ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_void_p)]),
    ("spec_pool_destroy", ctypes.c_int, [ctypes.c_void_p]),
    ("spec_pool_reserve", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int]),
    ("spec_pool_commit", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int, ctypes.c_int]),
    ("spec_pool_release", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("spec_pool_share", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int, ctypes.c_int32]),
    ("spec_pool_block_table", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P, ctypes.c_int, _I32P]),
    ("spec_pool_refcount", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("spec_pool_free_count", ctypes.c_int, [ctypes.c_void_p]),
]
EXPORTS = [s[0] for s in _SIGS]


def lib() -> ctypes.CDLL:
    """Load libspec.so (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with lossless_speculative_decoding_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in _SIGS:
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(rc: int) -> int:
    if rc < 0:
        raise SpecError(rc, lib().spec_last_error().decode())
    return rc


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


def _ptr(x) -> int:
    """Device pointer of a torch tensor or a raw integer address."""
    if x is None:
        return 0
    return int(x.data_ptr()) if hasattr(x, "data_ptr") else int(x)


def make_config(**kw) -> spec_config:
    c = spec_config()
    c.rope_theta, c.rms_eps = 10000.0, 1e-6
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def spec_tensor_count(cfg: spec_config) -> int:
    return _check(lib().spec_tensor_count(ctypes.byref(cfg)))


def spec_tensor_bytes(cfg: spec_config, index: int) -> int:
    return _check(lib().spec_tensor_bytes(ctypes.byref(cfg), index))


def spec_init_model(cfg: spec_config, host_tensors: Sequence[np.ndarray], cuda_stream: int = 0) -> int:
    n = spec_tensor_count(cfg)
    if len(host_tensors) != n:
        raise ValueError(f"expected {n} tensors, got {len(host_tensors)}")
    arrs = [np.ascontiguousarray(a) for a in host_tensors]
    for i, a in enumerate(arrs):
        want = spec_tensor_bytes(cfg, i)
        if a.nbytes != want:
            raise ValueError(f"tensor {i}: {a.nbytes} bytes, expected {want}")
    ptrs = (ctypes.c_void_p * n)(*[a.ctypes.data if a.nbytes else None for a in arrs])
    out = ctypes.c_void_p()
    _check(lib().spec_init_model(ctypes.byref(cfg), ptrs, cuda_stream, ctypes.byref(out)))
    return out.value


def spec_free_model(m: int) -> None:
    _check(lib().spec_free_model(m))


def spec_register_prefix(m: int, tokens) -> int:
    t = _i32(tokens)
    out = ctypes.c_int32()
    _check(lib().spec_register_prefix(m, _p(t), len(t), ctypes.byref(out)))
    return out.value


def spec_release_prefix(m: int, prefix_id: int) -> None:
    _check(lib().spec_release_prefix(m, prefix_id))


def spec_prefill(m: int, seq_id: int, prefix_id: int, vis_embeds_dev, n_vis: int, tokens) -> int:
    t = _i32(tokens if tokens is not None else [])
    out = ctypes.c_int32()
    _check(lib().spec_prefill(m, seq_id, prefix_id, _ptr(vis_embeds_dev), n_vis, _p(t), len(t), ctypes.byref(out)))
    return out.value


def spec_verify_step(m: int, seq_id: int, drafts) -> tuple:
    d = _i32(drafts)
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().spec_verify_step(m, seq_id, _p(d), len(d), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def spec_verify_step_batch(m: int, seq_ids, drafts, n_draft) -> tuple:
    s, d, n = _i32(seq_ids), _i32(drafts), _i32(n_draft)
    acc, bon = np.zeros(len(s), np.int32), np.zeros(len(s), np.int32)
    _check(lib().spec_verify_step_batch(m, len(s), _p(s), _p(d), _p(n), _p(acc), _p(bon)))
    return acc, bon


def spec_verify_step_sample_batch(m: int, seq_ids, drafts, n_draft, u_accept, u_sample,
                                  temperature: float) -> tuple:
    s, d, n = _i32(seq_ids), _i32(drafts), _i32(n_draft)
    ua = np.ascontiguousarray(u_accept, np.float32).reshape(-1)
    us = np.ascontiguousarray(u_sample, np.float32).reshape(-1)
    acc, tok = np.zeros(len(s), np.int32), np.zeros(len(s), np.int32)
    _check(lib().spec_verify_step_sample_batch(m, len(s), _p(s), _p(d), _p(n),
                                               ua.ctypes.data if ua.size else None, us.ctypes.data,
                                               float(temperature), _p(acc), _p(tok)))
    return acc, tok


def spec_verify_step_sample_dev(m: int, n_seq: int, seq_ids_dev, drafts_dev, n_draft_dev, u_accept_dev,
                                u_sample_dev, temperature: float, out_acc_dev, out_tok_dev) -> None:
    _check(lib().spec_verify_step_sample_dev(m, n_seq, _ptr(seq_ids_dev), _ptr(drafts_dev), _ptr(n_draft_dev),
                                             _ptr(u_accept_dev), _ptr(u_sample_dev), float(temperature),
                                             _ptr(out_acc_dev), _ptr(out_tok_dev)))


def spec_verify_step_batch_dev(m: int, n_seq: int, seq_ids_dev, drafts_dev, n_draft_dev, out_acc_dev,
                               out_bonus_dev) -> None:
    _check(lib().spec_verify_step_batch_dev(m, n_seq, _ptr(seq_ids_dev), _ptr(drafts_dev), _ptr(n_draft_dev),
                                            _ptr(out_acc_dev), _ptr(out_bonus_dev)))


def spec_reserve_seq(m: int, seq_id: int, n_tokens: int) -> None:
    _check(lib().spec_reserve_seq(m, seq_id, n_tokens))


def spec_sync_seqs(m: int) -> None:
    _check(lib().spec_sync_seqs(m))


def spec_release_seq(m: int, seq_id: int) -> None:
    _check(lib().spec_release_seq(m, seq_id))


def spec_seq_info(m: int, seq_id: int) -> tuple:
    n, g = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().spec_seq_info(m, seq_id, ctypes.byref(n), ctypes.byref(g)))
    return n.value, g.value


def spec_seq_tokens(m: int, seq_id: int) -> np.ndarray:
    _, n = spec_seq_info(m, seq_id)
    out = np.zeros(max(n, 1), np.int32)
    k = _check(lib().spec_seq_tokens(m, seq_id, _p(out), n))
    return out[:k]


def spec_seq_block_table(m: int, seq_id: int, cap: int = 4096) -> np.ndarray:
    out = np.full(cap, -1, np.int32)
    n = ctypes.c_int32()
    _check(lib().spec_seq_block_table(m, seq_id, _p(out), cap, ctypes.byref(n)))
    return out[:n.value]


def spec_free_pages(m: int) -> int:
    return _check(lib().spec_free_pages(m))


def spec_debug_logits(m: int, seq_ids, drafts, logits_dev) -> None:
    s, d = _i32(seq_ids), _i32(drafts)
    _check(lib().spec_debug_logits(m, len(s), _p(s), _p(d), _ptr(logits_dev)))


def spec_step_launches(m: int, n_seq: int) -> int:
    return _check(lib().spec_step_launches(m, n_seq))


def spec_mtp_init(m: int, host_tensors: Sequence[np.ndarray], inter: int) -> None:
    """host_tensors: the 13 arrays in the order of spec.h (encoded as stored)."""
    if len(host_tensors) != 13:
        raise ValueError(f"expected 13 tensors, got {len(host_tensors)}")
    arrs = [np.ascontiguousarray(a) for a in host_tensors]
    ptrs = (ctypes.c_void_p * 13)(*[a.ctypes.data for a in arrs])
    _check(lib().spec_mtp_init(m, ptrs, inter))


def spec_mtp_draft(m: int, seq_id: int, K: int) -> np.ndarray:
    out = np.zeros(K, np.int32)
    _check(lib().spec_mtp_draft(m, seq_id, K, _p(out)))
    return out


def spec_mtp_debug_draft(m: int, seq_id: int, K: int, logits_dev, states_dev, states_cap: int) -> tuple:
    """(drafts, number of state rows written)."""
    out = np.zeros(K, np.int32)
    n = ctypes.c_int32()
    _check(lib().spec_mtp_debug_draft(m, seq_id, K, _p(out), _ptr(logits_dev), _ptr(states_dev), states_cap,
                                      ctypes.byref(n)))
    return out, n.value


def spec_profile_steps_dev(m: int, n_seq: int, seq_ids_dev, drafts_dev, n_draft_dev, n_steps: int,
                           drafts_step_stride: int) -> dict:
    out = (spec_kernel_stat * SPEC_KCLASS_COUNT)()
    n = _check(lib().spec_profile_steps_dev(m, n_seq, _ptr(seq_ids_dev), _ptr(drafts_dev), _ptr(n_draft_dev),
                                            n_steps, drafts_step_stride, out, SPEC_KCLASS_COUNT))
    return {spec_kernel_class_name(i): dict(ms=out[i].ms, launches=out[i].launches, units=out[i].units)
            for i in range(n)}


def spec_kernel_class_name(cls: int) -> str:
    return lib().spec_kernel_class_name(cls).decode()


def spec_io_bytes(m: int) -> tuple:
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().spec_io_bytes(m, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def spec_lmhead_argmax_scratch_bytes(T: int, vocab: int) -> int:
    return _check(lib().spec_lmhead_argmax_scratch_bytes(T, vocab))


def spec_lmhead_argmax(x_dev, T: int, hidden: int, vocab: int, w_dev, w_dtype: int, gamma_dev, eps: float,
                       scratch_dev, scratch_bytes: int, out_tokens_dev, cuda_stream: int = 0) -> None:
    _check(lib().spec_lmhead_argmax(_ptr(x_dev), T, hidden, vocab, _ptr(w_dev), w_dtype, _ptr(gamma_dev), eps,
                                    _ptr(scratch_dev), scratch_bytes, _ptr(out_tokens_dev), cuda_stream))


SPEC_LMHEAD_NOALLOC_MAX_PAIRS = 262144


def spec_lmhead_argmax_noalloc(x_dev, T: int, hidden: int, vocab: int, w_dev, w_dtype: int, gamma_dev,
                               eps: float, out_tokens_dev, cuda_stream: int = 0) -> None:
    _check(lib().spec_lmhead_argmax_noalloc(_ptr(x_dev), T, hidden, vocab, _ptr(w_dev), w_dtype, _ptr(gamma_dev),
                                            eps, _ptr(out_tokens_dev), cuda_stream))


def spec_rejection_sample(logits_dev, drafts_dev, q_dev, u_accept_dev, u_sample_dev, n_seq: int, K: int,
                          vocab: int, temperature: float, out_accepted_dev, out_token_dev, cuda_stream: int = 0) -> None:
    _check(lib().spec_rejection_sample(_ptr(logits_dev), _ptr(drafts_dev), _ptr(q_dev), _ptr(u_accept_dev),
                                       _ptr(u_sample_dev), n_seq, K, vocab, float(temperature),
                                       _ptr(out_accepted_dev), _ptr(out_token_dev), cuda_stream))


def spec_rejection_sample_ws_bytes(n_seq: int, K: int) -> int:
    return _check(lib().spec_rejection_sample_ws_bytes(n_seq, K))


def spec_rejection_sample_ws(logits_dev, drafts_dev, q_dev, u_accept_dev, u_sample_dev, n_seq: int, K: int,
                             vocab: int, temperature: float, out_accepted_dev, out_token_dev, ws_dev, ws_bytes: int,
                             cuda_stream: int = 0) -> None:
    _check(lib().spec_rejection_sample_ws(_ptr(logits_dev), _ptr(drafts_dev), _ptr(q_dev), _ptr(u_accept_dev),
                                          _ptr(u_sample_dev), n_seq, K, vocab, float(temperature),
                                          _ptr(out_accepted_dev), _ptr(out_token_dev), _ptr(ws_dev), ws_bytes,
                                          cuda_stream))


def spec_tc_gemm_test(a_dev, a2_dev, b_dev, b_lo_dev, M: int, N: int, K: int, dual: int, out_dev, err_dev,
                      cuda_stream: int = 0, a_scale_dev=None, a2_scale_dev=None, a_fp8: bool = False,
                      n_tile: int = 0, k_split: int = 1, flags: int = 0) -> None:
    _check(lib().spec_tc_gemm_test(_ptr(a_dev), _ptr(a2_dev), _ptr(a_scale_dev), _ptr(a2_scale_dev), int(a_fp8),
                                   _ptr(b_dev), _ptr(b_lo_dev), M, N, K, dual, n_tile, k_split, flags,
                                   _ptr(out_dev), _ptr(err_dev), cuda_stream))


def spec_strerror(code: int) -> str:
    return lib().spec_strerror(code).decode()


# ---- host-only allocator ----------------------------------------------------
def spec_pool_create(n_pages: int, page_size: int, max_seqs: int, max_pages_per_seq: int) -> int:
    out = ctypes.c_void_p()
    _check(lib().spec_pool_create(n_pages, page_size, max_seqs, max_pages_per_seq, ctypes.byref(out)))
    return out.value


def spec_pool_destroy(p: int) -> None:
    _check(lib().spec_pool_destroy(p))


def spec_pool_reserve(p: int, seq: int, n_tokens: int) -> int:
    return lib().spec_pool_reserve(p, seq, n_tokens)


def spec_pool_commit(p: int, seq: int, new_len: int, keep_pages: int = 0) -> int:
    return lib().spec_pool_commit(p, seq, new_len, keep_pages)


def spec_pool_release(p: int, seq: int) -> int:
    return lib().spec_pool_release(p, seq)


def spec_pool_share(p: int, src: int, n_pages: int, dst: int) -> int:
    return lib().spec_pool_share(p, src, n_pages, dst)


def spec_pool_block_table(p: int, seq: int, cap: int = 4096) -> list:
    out = np.zeros(cap, np.int32)
    n = ctypes.c_int32()
    _check(lib().spec_pool_block_table(p, seq, _p(out), cap, ctypes.byref(n)))
    return out[:n.value].tolist()


def spec_pool_refcount(p: int, page: int) -> int:
    return lib().spec_pool_refcount(p, page)


def spec_pool_free_count(p: int) -> int:
    return lib().spec_pool_free_count(p)
