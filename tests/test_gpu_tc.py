"""Tensor-core GEMM (tcgen05, TMA-staged, TMEM accumulator) against a plain
float64 matmul of the same bf16 values: the store epilogue (fp32 out) and
the dual SwiGLU epilogue (bf16 out), over shapes with partial activation
boxes, more K tiles than pipeline stages, several column tiles, CTAs of 1 to
4 activation boxes (MMA N of 32 to 256 with the hi and lo rows) and one- and
two-atom stages with an odd number of K atoms; and the
hi + lo split of fp32 activations, which must reach near-fp32 accuracy (a
bound a single bf16 operand misses by two orders of magnitude)."""
import numpy as np
import pytest

import synthetic as syn
import oracle

pytestmark = pytest.mark.gpu


def _f16_parts(x):
    """f16 hi + lo parts of 256 x (the operand form of the e4m3-weight GEMMs),
    as int16 bit patterns: lo is the f16 rounding of what hi leaves."""
    y = x.astype(np.float32) * np.float32(256.0)
    hi = y.astype(np.float16)
    lo = (y - hi.astype(np.float32)).astype(np.float16)
    return hi.view(np.int16), lo.view(np.int16)


def _bf16(rng, shape, scale):
    bits = syn.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))
    return bits, oracle.decode_bf16(bits)


@pytest.mark.parametrize("M,N,K", [(128, 32, 64), (256, 40, 320), (384, 300, 1280), (128, 1, 896), (128, 96, 1344)])
def test_tc_gemm_store(M, N, K):
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(M + N + K)
    ab, af = _bf16(rng, (M, K), 0.05)
    bb, bf = _bf16(rng, (N, K), 1.0)
    a = torch.from_numpy(ab.view(np.int16)).cuda()
    b = torch.from_numpy(bb.view(np.int16)).cuda()
    out = torch.full((N, M), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.spec_tc_gemm_test(a, None, b, None, M, N, K, 0, out, err, 0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = bf.astype(np.float64) @ af.astype(np.float64).T
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-4, atol=1e-4 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K", [(256, 48, 192), (128, 256, 1280)])
def test_tc_gemm_swiglu(M, N, K):
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(7 * M + N)
    gb, gf = _bf16(rng, (M, K), 0.05)
    ub, uf = _bf16(rng, (M, K), 0.05)
    bb, bf = _bf16(rng, (N, K), 1.0)
    g = torch.from_numpy(gb.view(np.int16)).cuda()
    u = torch.from_numpy(ub.view(np.int16)).cuda()
    b = torch.from_numpy(bb.view(np.int16)).cuda()
    out = torch.zeros((N, M), dtype=torch.int16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.spec_tc_gemm_test(g, u, b, None, M, N, K, 1, out, err, 0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    gg = bf.astype(np.float64) @ gf.astype(np.float64).T
    uu = bf.astype(np.float64) @ uf.astype(np.float64).T
    ref = gg / (1 + np.exp(-gg)) * uu
    got = oracle.decode_bf16(out.cpu().numpy().view(np.uint16)).astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-2, atol=1e-2 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K,nt", [(256, 300, 512, 0), (128, 9, 2048, 0), (256, 300, 512, 32), (384, 100, 768, 64),
                                     (128, 80, 640, 0), (256, 96, 1344, 0)])
def test_tc_gemm_split_activations(M, N, K, nt):
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(11 * M + N)
    ab, af = _bf16(rng, (M, K), 0.05)
    x = rng.standard_normal((N, K)).astype(np.float32)
    hi = syn.f32_to_bf16_bits(x)
    lo = syn.f32_to_bf16_bits((x - oracle.decode_bf16(hi)).astype(np.float32))
    a = torch.from_numpy(ab.view(np.int16)).cuda()
    bh = torch.from_numpy(hi.view(np.int16)).cuda()
    bl = torch.from_numpy(lo.view(np.int16)).cuda()
    out = torch.full((N, M), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.spec_tc_gemm_test(a, None, bh, bl, M, N, K, 0, out, err, 0, n_tile=nt)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = x.astype(np.float64) @ af.astype(np.float64).T
    got = out.cpu().numpy()
    # hi + lo carries ~16 mantissa bits (relative residual <= 2^-17); bf16
    # alone would leave errors near 2^-9 of the row scale
    np.testing.assert_allclose(got, ref, rtol=0, atol=5e-5 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K,dual,nt", [(256, 40, 320, 0, 0), (128, 200, 1280, 0, 32), (256, 48, 192, 1, 0),
                                           (128, 130, 896, 1, 32), (128, 90, 704, 0, 0), (128, 70, 448, 1, 0)])
def test_tc_gemm_fp8_weights(M, N, K, dual, nt):
    """e4m3 weights widened to f16 in shared memory, activations as f16 hi + lo
    parts of 256 x, per-row scales (and the 1/256) applied in the epilogue:
    against float64 of the decoded e4m3 values times the scales."""
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(5 * M + N + dual)

    def q8(shape):
        w = (rng.standard_normal(shape) * 0.05).astype(np.float32)
        codes, sc = syn.quantize_rows_e4m3(w)
        return codes, sc, oracle.decode_e4m3(codes).astype(np.float64) * sc[:, None].astype(np.float64)

    c1, s1, w1 = q8((M, K))
    c2, s2, w2 = q8((M, K))
    x = rng.standard_normal((N, K)).astype(np.float32)
    hi, lo = _f16_parts(x)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    a, a2, sa, sa2 = dev(c1.view(np.int8)), dev(c2.view(np.int8)), dev(s1), dev(s2)
    bh, bl = dev(hi.view(np.int16)), dev(lo.view(np.int16))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if dual:
        out = torch.zeros((N, M), dtype=torch.int16, device="cuda")
        B.spec_tc_gemm_test(a, a2, bh, bl, M, N, K, 1, out, err, 0, a_scale_dev=sa, a2_scale_dev=sa2, a_fp8=True,
                            n_tile=nt)
    else:
        out = torch.full((N, M), float("nan"), device="cuda")
        B.spec_tc_gemm_test(a, None, bh, bl, M, N, K, 0, out, err, 0, a_scale_dev=sa, a_fp8=True, n_tile=nt)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    xf = x.astype(np.float64)
    if dual:
        gg, uu = xf @ w1.T, xf @ w2.T
        ref = gg / (1 + np.exp(-gg)) * uu
        got = out.cpu().numpy().view(np.float16).astype(np.float64) / 256.0
        np.testing.assert_allclose(got, ref, rtol=2e-3, atol=2e-3 * np.abs(ref).max())
    else:
        ref = xf @ w1.T
        np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=5e-5 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K,dual,ks,fp8", [(256, 40, 1280, 0, 4, 0), (128, 300, 2048, 0, 8, 0), (256, 48, 1280, 1, 3, 0),
                                               (128, 33, 1280, 0, 5, 1), (128, 64, 640, 1, 2, 1)])
def test_tc_gemm_split_k(M, N, K, dual, ks, fp8):
    """K split across CTAs: each split's fp32 partial is stored and the tile's
    last split adds them in split order, then runs the store / SwiGLU epilogue."""
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(13 * M + N + ks)
    if fp8:
        def mat():
            w = (rng.standard_normal((M, K)) * 0.05).astype(np.float32)
            codes, sc = syn.quantize_rows_e4m3(w)
            return codes.view(np.int8), sc, oracle.decode_e4m3(codes).astype(np.float64) * sc[:, None]
    else:
        def mat():
            bits, f = _bf16(rng, (M, K), 0.05)
            return bits.view(np.int16), None, f.astype(np.float64)
    a, sa, w1 = mat()
    a2, sa2, w2 = mat()
    x = rng.standard_normal((N, K)).astype(np.float32)
    if fp8:
        hi, lo = _f16_parts(x)
    else:
        hi = syn.f32_to_bf16_bits(x)
        lo = syn.f32_to_bf16_bits((x - oracle.decode_bf16(hi)).astype(np.float32))
    dev = lambda v: None if v is None else torch.from_numpy(np.ascontiguousarray(v)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xf = x.astype(np.float64)
    if dual:
        out = torch.zeros((N, M), dtype=torch.int16, device="cuda")
        B.spec_tc_gemm_test(dev(a), dev(a2), dev(hi.view(np.int16)), dev(lo.view(np.int16)), M, N, K, 1, out, err, 0,
                            a_scale_dev=dev(sa), a2_scale_dev=dev(sa2), a_fp8=bool(fp8), k_split=ks)
        torch.cuda.synchronize()
        gg, uu = xf @ w1.T, xf @ w2.T
        ref = gg / (1 + np.exp(-gg)) * uu
        if fp8:
            got = out.cpu().numpy().view(np.float16).astype(np.float64) / 256.0
        else:
            got = oracle.decode_bf16(out.cpu().numpy().view(np.uint16)).astype(np.float64)
        np.testing.assert_allclose(got, ref, rtol=1e-2, atol=1e-2 * np.abs(ref).max())
    else:
        out = torch.full((N, M), float("nan"), device="cuda")
        B.spec_tc_gemm_test(dev(a), None, dev(hi.view(np.int16)), dev(lo.view(np.int16)), M, N, K, 0, out, err, 0,
                            a_scale_dev=dev(sa), a_fp8=bool(fp8), k_split=ks)
        torch.cuda.synchronize()
        ref = xf @ w1.T
        np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=5e-5 * np.abs(ref).max())
    assert int(err.item()) == 0


def test_wait_deadline_reports_timeout_and_context_survives():
    """Every mbarrier wait of the tensor-core GEMM ends by a deadline read from
    %globaltimer. With the test-only stall flag the kernel issues no loads, so
    its waits must run out: the call returns within a few deadlines, the
    timeout bit (8) is set, the output is untouched, and the next normal GEMM
    on the same context is correct."""
    import time
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    M, N, K = 256, 32, 512
    rng = np.random.default_rng(41)
    a = torch.from_numpy(syn.f32_to_bf16_bits((rng.standard_normal((M, K)) * 0.05).astype(np.float32))
                         .view(np.int16)).cuda()
    x = torch.from_numpy(syn.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32)).view(np.int16)).cuda()
    out = torch.full((N, M), 7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    B.spec_tc_gemm_test(a, None, x, None, M, N, K, 0, out, err, 0, flags=1)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(err.item()) & 8, "the stalled kernel did not report a timeout"
    assert dt < 5.0, f"the stalled kernel took {dt:.2f} s to give up"
    assert bool((out == 7.0).all()), "a stalled kernel wrote results"
    err.zero_()
    B.spec_tc_gemm_test(a, None, x, None, M, N, K, 0, out, err, 0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.decode_bf16(x.cpu().numpy().view(np.uint16)) @ oracle.decode_bf16(a.cpu().numpy().view(np.uint16)).T
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)
