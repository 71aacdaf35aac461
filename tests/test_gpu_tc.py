"""Tensor-core GEMM (tcgen05, TMA-staged, TMEM accumulator) against a plain
float64 matmul of the same bf16 values: the store epilogue (fp32 out) and
the dual SwiGLU epilogue (bf16 out), over shapes with partial activation
boxes, more K tiles than pipeline stages, and two column tiles."""
import numpy as np
import pytest

import synthetic as syn
import oracle

pytestmark = pytest.mark.gpu


def _bf16(rng, shape, scale):
    bits = syn.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))
    return bits, oracle.decode_bf16(bits)


@pytest.mark.parametrize("M,N,K", [(128, 32, 64), (256, 40, 320), (384, 300, 1280), (128, 1, 896)])
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
    B.spec_tc_gemm_test(a, None, b, M, N, K, 0, out, err, 0)
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
    B.spec_tc_gemm_test(g, u, b, M, N, K, 1, out, err, 0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    gg = bf.astype(np.float64) @ gf.astype(np.float64).T
    uu = bf.astype(np.float64) @ uf.astype(np.float64).T
    ref = gg / (1 + np.exp(-gg)) * uu
    got = oracle.decode_bf16(out.cpu().numpy().view(np.uint16)).astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-2, atol=1e-2 * np.abs(ref).max())
