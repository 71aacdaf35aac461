"""The allocation-free LM-head entry point, for callers that cannot allocate
device memory while they run (no cudaMalloc by them or by the library): it
must give exactly the tokens of the entry point that takes caller scratch,
on consecutive calls that share its fixed device array. Collected last so a
run that stops at the first failure has run every other test first."""
import numpy as np
import pytest

import synthetic as syn

pytestmark = pytest.mark.gpu


def test_noalloc_lmhead_matches_scratch_entry():
    import torch
    from lossless_speculative_decoding_gb300 import build
    build.build()
    from lossless_speculative_decoding_gb300 import binding as B
    torch.cuda.set_device(0)
    rng = np.random.default_rng(11)
    # two calls in a row with different shapes and inputs: the shared array
    # keeps the first call's candidates, which the second must not pick up
    for T, h, V in [(4, 1280, 129280), (3, 256, 1000)]:
        x = torch.from_numpy(rng.standard_normal((T, h)).astype(np.float32)).cuda()
        wbits = syn.f32_to_bf16_bits((rng.standard_normal((V, h)) * 0.02).astype(np.float32))
        w = torch.from_numpy(wbits.view(np.int16)).cuda()
        gamma = torch.from_numpy((1 + 0.1 * rng.standard_normal(h)).astype(np.float32)).cuda()
        nbytes = B.spec_lmhead_argmax_scratch_bytes(T, V)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        ref = torch.full((T,), -1, dtype=torch.int32, device="cuda")
        got = torch.full((T,), -2, dtype=torch.int32, device="cuda")
        B.spec_lmhead_argmax(x, T, h, V, w, syn.BF16, gamma, 1e-6, scratch, nbytes, ref, 0)
        B.spec_lmhead_argmax_noalloc(x, T, h, V, w, syn.BF16, gamma, 1e-6, got, 0)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy())
        assert (ref.cpu().numpy() >= 0).all()
        # a warm call takes no device memory: the device's free bytes (as the
        # driver reports them, whatever torch's allocator caches) do not move
        free0 = torch.cuda.mem_get_info()[0]
        B.spec_lmhead_argmax_noalloc(x, T, h, V, w, syn.BF16, gamma, 1e-6, got, 0)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy())


def test_noalloc_rejects_oversize():
    import torch
    from lossless_speculative_decoding_gb300 import build
    build.build()
    from lossless_speculative_decoding_gb300 import binding as B
    torch.cuda.set_device(0)
    T, h, V = 64, 256, 151936            # 64 * 4748 candidates > the fixed array
    x = torch.zeros((T, h), device="cuda")
    w = torch.zeros((V, h), dtype=torch.int16, device="cuda")
    out = torch.zeros(T, dtype=torch.int32, device="cuda")
    with pytest.raises(B.SpecError) as e:
        B.spec_lmhead_argmax_noalloc(x, T, h, V, w, syn.BF16, torch.ones(h, device="cuda"), 1e-6, out, 0)
    assert e.value.code == -1 and "SPEC_LMHEAD_NOALLOC_MAX_PAIRS" in str(e.value)
