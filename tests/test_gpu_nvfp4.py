"""GPU parity of NVFP4-weight models ("OCRia-1 technical report guide",
inference stack: NVFP4 weights) against the oracle, which decodes every
record to fp32 (e2m1 * e4m3 block scale * fp32 matrix scale).

Same bar as the bf16 and e4m3 models: verify-row logits within 2e-2 of the
oracle row's range, tokens equal to the oracle's except at oracle margins
below 1e-3 (counted), accepted length and bonus bit-exact for the GPU's
argmaxes, speculative == greedy on the GPU."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _util import gpu_model, margin_exempt, row_tol_ok

pytestmark = pytest.mark.gpu

MOE_SMALL_Q4 = syn.scaled(syn.MOE3B, name="moe-small-nvfp4", n_layers=2, hidden=256, n_q_heads=2, n_kv_heads=2,
                          head_dim=128, n_experts=16, top_k=4, n_shared=2, inter=128, vocab=2048, wdtype=syn.NVFP4)
DENSE_SMALL_Q4 = syn.scaled(syn.DENSE4B, name="dense-small-gqa-nvfp4", n_layers=2, hidden=256, n_q_heads=8,
                            n_kv_heads=2, head_dim=64, inter=512, vocab=2048, wdtype=syn.NVFP4)


@pytest.mark.parametrize("cfg,K", [(MOE_SMALL_Q4, 3), (DENSE_SMALL_Q4, 7)])
def test_nvfp4_parity(cfg, K):
    w = syn.generate_weights(cfg, 7)
    om = oracle.OracleModel(w)
    wl = syn.Workload("t", cfg, 1, K, "iid", 0.6, (96, 0, 0), 8, 0, (48,))
    prompt = syn.make_prompts(wl)[0]
    gm = gpu_model(cfg, w, max_ctx=512, max_draft=K)
    first = gm.prefill(0, prompt.visual, prompt.tokens)
    cache = oracle.KVCache(cfg)
    lg0 = oracle.forward(om, cache, oracle.prompt_embeddings(om, prompt), np.arange(prompt.length))[-1]
    assert first == int(np.argmax(lg0)) or margin_exempt(lg0)
    rng = np.random.default_rng(3)
    toks = [first]
    n_rows = n_exempt = 0
    worst = 0.0
    for step in range(6):
        d = [int(t) for t in rng.integers(0, cfg.vocab, K)]
        lg = gm.debug_logits([0], np.array(d))
        base = cache.length
        ol = oracle.verify_rows(om, cache, toks[-1], d)
        ok = row_tol_ok(lg, ol, 2e-2)
        assert ok.all(), np.abs(lg - ol).max(-1) / (ol.max(-1) - ol.min(-1))
        worst = max(worst, float((np.abs(lg - ol).max(-1) / (ol.max(-1) - ol.min(-1))).max()))
        n_rows += len(ok)
        g_gpu, g_or = np.argmax(lg, -1), np.argmax(ol, -1)
        for i in np.nonzero(g_gpu != g_or)[0]:
            assert margin_exempt(ol[i]), f"token mismatch at row {i} outside a near-tie"
            n_exempt += 1
        a, b = gm.verify(0, d)
        assert (a, b) == oracle.accept(d, g_gpu)
        cache.truncate(base + a + 1)
        toks += d[:a] + [b]
    gm.close()
    print(f"nvfp4 parity {cfg.name}: rows {n_rows}, margin-exempt tokens {n_exempt}, max err {worst:.3g} of range")


def test_nvfp4_speculative_equals_greedy():
    cfg = MOE_SMALL_Q4
    w = syn.generate_weights(cfg, 5)
    wl = syn.Workload("t", cfg, 1, 3, "iid", 0.6, (32, 0, 0), 6, 0, (40,))
    p = syn.make_prompts(wl)[0]
    gm = gpu_model(cfg, w, max_ctx=256, max_draft=3)
    greedy = [gm.prefill(0, p.visual, p.tokens)]
    while len(greedy) < 40:
        greedy.append(gm.verify(0, [])[1])
    gm.release(0)
    drafter = syn.Drafter("iid", 0.6, cfg.vocab, seed=4)
    spec = [gm.prefill(0, p.visual, p.tokens)]
    step = 0
    while len(spec) < 40:
        m = min(3, 40 - len(spec) - 1)
        d = [int(x) for x in drafter.propose(greedy, len(spec), m, 0, step)]
        a, b = gm.verify(0, d)
        spec += d[:a] + [b]
        step += 1
    gm.close()
    assert spec[:40] == greedy


def test_nvfp4_shape_limits():
    from lossless_speculative_decoding_gb300 import binding as B
    w = syn.generate_weights(MOE_SMALL_Q4, 1)
    with pytest.raises(B.SpecError) as e:             # 2 x 8 rows a step: the tensor-core path
        gpu_model(MOE_SMALL_Q4, w, max_ctx=256, max_draft=7, max_seqs=2, max_batch=2)
    assert e.value.code == B.SPEC_ERR_UNSUPPORTED
    odd = syn.scaled(MOE_SMALL_Q4, name="odd", inter=192)
    with pytest.raises(B.SpecError) as e:
        gpu_model(odd, syn.generate_weights(odd, 1), max_ctx=256, max_draft=3)
    assert e.value.code == B.SPEC_ERR_UNSUPPORTED
