"""Pins of the rejection-sampling oracle (oracle/sampling.py) against what the
mathematics fixes: the acceptance probability min(1, p/q), the residual
distribution max(0, p - q) / S, the composed law of the first emitted token
(exactly p -- the losslessness the end-to-end OCR explainer states in section
6.1 and section 11), its greedy limit (the already-pinned greedy acceptance
rule) and the q = p special case. Exact probabilities come from evaluating the
oracle on grids of uniforms: every decision is a threshold in one uniform, so
a grid of N cell midpoints measures each outcome to within 1/N per threshold."""
import numpy as np
import pytest

import oracle
from oracle import sampling as smp

N = 2000
GRID = (np.arange(N) + 0.5) / N


def _case(seed, V=6):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((2, V)) * 1.5
    q = rng.dirichlet(np.ones(V) * 0.7, size=1)
    return logits, q


def test_inverse_cdf_edges():
    w = np.array([0.0, 1.0, 0.0, 3.0])
    assert smp.inverse_cdf(w, 0.0)[0] == 1          # zero-weight tokens are never drawn
    assert smp.inverse_cdf(w, 0.2)[0] == 1          # target 0.8 < 1
    assert smp.inverse_cdf(w, 0.25)[0] == 3         # target 1.0: first cumulative value > 1.0
    assert smp.inverse_cdf(w, 0.999)[0] == 3


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_acceptance_probability_is_min_one_p_over_q(seed):
    logits, q = _case(seed)
    p = smp.target_probs(logits[0], 1.0)
    for d in range(len(p)):
        acc = np.mean([smp.rejection_sample(logits, [d], q, [u], [0.5, 0.5])[0] == 1 for u in GRID])
        assert abs(acc - min(1.0, p[d] / q[0][d])) <= 1.0 / N + 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_residual_distribution(seed):
    logits, q = _case(seed)
    p = smp.target_probs(logits[0], 1.0)
    r = np.maximum(p - q[0], 0.0)
    for d in np.nonzero(p < q[0])[0]:                  # drafts that can be rejected
        toks = np.array([smp.rejection_sample(logits, [d], q, [1.0 - 1e-9], [u, 0.5])[1] for u in GRID])
        assert (toks != d).all()                        # the rejected draft has no residual mass
        freq = np.bincount(toks, minlength=len(p)) / N
        np.testing.assert_allclose(freq, r / r.sum(), atol=1.0 / N + 1e-12)


@pytest.mark.parametrize("seed", [3, 4, 5, 6])
def test_first_token_is_distributed_as_the_target(seed):
    """P(first emitted token = v) = sum_d q(d) [P(acc | d) 1{v = d} + P(rej | d) R_d(v)] = p(v)."""
    logits, q = _case(seed)
    V = logits.shape[1]
    p = smp.target_probs(logits[0], 1.0)
    law = np.zeros(V)
    for d in range(V):
        acc = np.mean([smp.rejection_sample(logits, [d], q, [u], [0.5, 0.5])[0] == 1 for u in GRID])
        law[d] += q[0][d] * acc
        if acc < 1.0:
            toks = [smp.rejection_sample(logits, [d], q, [1.0 - 1e-9], [u, 0.5])[1] for u in GRID]
            law += q[0][d] * (1.0 - acc) * np.bincount(toks, minlength=V) / N
    np.testing.assert_allclose(law, p, atol=(V + 1) / N)
    # a plausible mistake (accepting with probability p instead of min(1, p/q))
    # is far outside that bound
    wrong = np.zeros(V)
    for d in range(V):
        a = p[d]
        r = np.maximum(p - q[0], 0.0)
        wrong[d] += q[0][d] * a
        wrong += q[0][d] * (1 - a) * r / r.sum()
    assert np.abs(wrong - p).max() > 10 * (V + 1) / N


@pytest.mark.parametrize("seed", [7, 8, 9])
def test_certain_drafter_is_lossless_for_any_draft_law(seed):
    """q = None (a drafter certain of its drafts, the form the model's sampled
    step uses) with drafts drawn from an arbitrary law r: P(first emitted = v)
    = sum_d r(d) [p(d) 1{v = d} + (1 - p(d)) p(v) 1{v != d} / (1 - p(d))] = p(v)."""
    logits, _ = _case(seed)
    V = logits.shape[1]
    r = np.random.default_rng(seed + 100).dirichlet(np.ones(V) * 0.5)
    p = smp.target_probs(logits[0], 1.0)
    law = np.zeros(V)
    for d in range(V):
        acc = np.mean([smp.rejection_sample(logits, [d], None, [u], [0.5, 0.5])[0] == 1 for u in GRID])
        assert abs(acc - p[d]) <= 1.0 / N + 1e-12            # accepted with probability p(d)
        law[d] += r[d] * acc
        toks = [smp.rejection_sample(logits, [d], None, [1.0 - 1e-9], [u, 0.5])[1] for u in GRID]
        assert d not in toks                                   # the rejected draft is never drawn
        law += r[d] * (1.0 - acc) * np.bincount(toks, minlength=V) / N
    np.testing.assert_allclose(law, p, atol=(V + 1) / N)
    # a plausible mistake (the residual drawn from p itself, keeping the
    # rejected draft: law p(v) (r(v) + 1 - E_r[p])) lies well outside that bound
    wrong = np.zeros(V)
    for d in range(V):
        wrong[d] += r[d] * p[d]
        wrong += r[d] * (1.0 - p[d]) * p
    assert np.abs(wrong - p).max() > 5 * (V + 1) / N


def test_greedy_limit_is_the_greedy_rule():
    """With one-hot targets (logit gaps far beyond the float64 exponent range at
    this temperature) the rule reduces to the longest-prefix greedy acceptance
    for any drafts and any uniforms, with one-hot or certain drafters."""
    rng = np.random.default_rng(7)
    V, K = 50, 5
    for trial in range(200):
        g = rng.integers(0, V, K + 1)
        logits = rng.standard_normal((K + 1, V))
        logits[np.arange(K + 1), g] += 100.0
        drafts = [int(g[j]) if rng.random() < 0.6 else int(rng.integers(0, V)) for j in range(K)]
        ua, us = rng.random(K), rng.random(K + 1)
        assert smp.rejection_sample(logits, drafts, None, ua, us, temperature=0.05) == oracle.accept(drafts, g)


def test_q_equal_to_p_accepts_every_draft():
    rng = np.random.default_rng(8)
    V, K = 40, 3
    for trial in range(100):
        logits = rng.standard_normal((K + 1, V)) * 2
        q = np.stack([smp.target_probs(logits[j], 0.7) for j in range(K)])
        drafts = [int(rng.choice(V, p=q[j])) for j in range(K)]
        us = rng.random(K + 1)
        a, t = smp.rejection_sample(logits, drafts, q, rng.random(K), us, temperature=0.7)
        assert a == K
        assert t == smp.inverse_cdf(smp.target_probs(logits[K], 0.7), us[K])[0]


def test_sampling_loop_at_zero_temperature_is_greedy_decoding():
    """At a temperature far below the logit gaps every p_j is one-hot at the
    target's argmax, so the stochastic loop commits exactly greedy decoding,
    whatever the drafts and uniforms."""
    import synthetic as syn
    wl = syn.WORKLOADS["tiny_fp32_b1"]
    m = oracle.OracleModel(syn.generate_weights(wl.model, 0))
    prompt = syn.make_prompts(wl)[0]
    ref = oracle.greedy_decode(m, prompt, 20)
    drng = np.random.default_rng(3)

    def propose(out, k):                    # a certain drafter: right 60% of the time
        n = len(out)
        return [int(ref[n + j]) if n + j < len(ref) and drng.random() < 0.6 else int(drng.integers(0, 1024))
                for j in range(k)], None

    toks = smp.spec_sample_decode(m, prompt, 20, 3, propose, 1e-6, np.random.default_rng(4))
    assert np.array_equal(toks, ref)
