"""Kernel-level parity of the LM-head + argmax entry point against a plain
float32 restatement on the CPU (RMSNorm, matmul, argmax with the lowest index
on ties), at small shapes with a ragged vocabulary tail and at the 3B-MoE
shape."""
import numpy as np
import pytest

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu


def _ref_tokens(x, w, gamma, eps):
    u = oracle.rms_norm(x, gamma, eps)
    lg = u @ w.T
    return np.argmax(lg, -1), lg


@pytest.mark.parametrize("T,h,V,dt", [(1, 256, 1024, syn.F32), (4, 256, 1028, syn.BF16), (7, 128, 36, syn.F32),
                                      (4, 1280, 129280, syn.BF16), (32, 2560, 4096, syn.BF16)])
def test_lmhead_argmax_parity(T, h, V, dt):
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(T * 7 + h)
    x = rng.standard_normal((T, h)).astype(np.float32)
    w = (rng.standard_normal((V, h)) * 0.02).astype(np.float32)
    gamma = (1 + 0.1 * rng.standard_normal(h)).astype(np.float32)
    if dt == syn.BF16:
        wbits = syn.f32_to_bf16_bits(w)
        w = oracle.decode_bf16(wbits)
        w_dev = torch.from_numpy(wbits.view(np.int16)).cuda()
    else:
        w_dev = torch.from_numpy(w).cuda()
    x_dev, g_dev = torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda()
    nbytes = B.spec_lmhead_argmax_scratch_bytes(T, V)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    B.spec_lmhead_argmax(x_dev, T, h, V, w_dev, dt, g_dev, 1e-6, scratch, nbytes, out, 0)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref, lg = _ref_tokens(x, w, gamma, 1e-6)
    for t in np.nonzero(got != ref)[0]:
        s = np.sort(lg[t])
        assert s[-1] - s[-2] < 1e-3 * max(1.0, abs(s[-1])), (t, got[t], ref[t])


def test_lmhead_argmax_ties_lowest_index():
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    T, h, V = 2, 64, 512
    w = np.zeros((V, h), np.float32)
    w[[37, 300, 511], 0] = 1.0                                 # three equal maxima
    x = np.ones((T, h), np.float32)
    nbytes = B.spec_lmhead_argmax_scratch_bytes(T, V)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    B.spec_lmhead_argmax(torch.from_numpy(x).cuda(), T, h, V, torch.from_numpy(w).cuda(), syn.F32,
                         torch.ones(h, device="cuda"), 1e-6, scratch, nbytes, out, 0)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [37, 37]
    with pytest.raises(B.SpecError):
        B.spec_lmhead_argmax(torch.from_numpy(x).cuda(), T, h, V, torch.from_numpy(w).cuda(), syn.F32,
                             torch.ones(h, device="cuda"), 1e-6, scratch, nbytes - 8, out, 0)


def test_lmhead_argmax_nan_rows_give_valid_index():
    """A NaN logit ranks below every number: a row of NaNs yields index 0 (the
    lowest), and a NaN among numbers never wins, on both the scratch and the
    allocation-free entry points."""
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    T, h, V = 3, 256, 4096
    rng = np.random.default_rng(31)
    x = rng.standard_normal((T, h)).astype(np.float32)
    x[0, 5] = np.nan                                           # row 0: every logit NaN
    w = (rng.standard_normal((V, h)) * 0.02).astype(np.float32)
    w[[7, 2000], :] = np.nan                                   # two NaN vocabulary rows
    gamma = np.ones(h, np.float32)
    ref = np.argmax(np.where(np.isnan(_ref_tokens(x, w, gamma, 1e-6)[1]), -np.inf,
                             _ref_tokens(x, w, gamma, 1e-6)[1]), -1)
    ref[0] = 0
    nbytes = B.spec_lmhead_argmax_scratch_bytes(T, V)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for noalloc in (False, True):
        out = torch.full((T,), -1, dtype=torch.int32, device="cuda")
        args = (torch.from_numpy(x).cuda(), T, h, V, torch.from_numpy(w).cuda(), syn.F32,
                torch.from_numpy(gamma).cuda(), 1e-6)
        if noalloc:
            B.spec_lmhead_argmax_noalloc(*args, out, 0)
        else:
            B.spec_lmhead_argmax(*args, scratch, nbytes, out, 0)
        torch.cuda.synchronize()
        assert out.cpu().tolist() == ref.tolist()
