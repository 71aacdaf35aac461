"""Rejection-sampling verification on the GPU (spec_rejection_sample) against
the oracle (oracle/sampling.py) and against the law it must produce.

* Parity: the same logits, drafts, drafter distributions and uniforms give the
  oracle's (accepted, token) exactly, except where the oracle's float64
  decision lies within 1e-4 (relative) of its threshold -- the device decides
  in float32 with its own summation order, so such a decision may go either
  way. Those cases are counted and must stay rare.
* Law: with drafts really drawn from q, the first and second emitted tokens of
  200,000 sequences are distributed as p_1 and p_2 (chi-square), the
  losslessness of the end-to-end OCR explainer, section 6.1 and section 11.
* Greedy limit: one-hot targets give the greedy acceptance rule exactly."""
import numpy as np
import pytest

import oracle
from oracle import sampling as smp

pytestmark = pytest.mark.gpu

TIE = 1e-4


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(logits, drafts, q, ua, us, temperature):
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    n, K1, V = logits.shape
    acc = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    B.spec_rejection_sample(_dev(logits.astype(np.float32)), _dev(drafts.astype(np.int32)) if K1 > 1 else None,
                            None if q is None else _dev(q.astype(np.float32)),
                            _dev(ua.astype(np.float32)) if K1 > 1 else None, _dev(us.astype(np.float32)),
                            n, K1 - 1, V, temperature, acc, tok, 0)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), tok.cpu().numpy()


def _inputs(rng, n, K, V, with_q, scale=3.0):
    logits = (rng.standard_normal((n, K + 1, V)) * scale).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.3, size=(n, K)).astype(np.float32) if with_q else None
    drafts = np.zeros((n, K), np.int64)
    for s in range(n):
        for j in range(K):
            if with_q:
                c = np.cumsum(q[s, j].astype(np.float64))
                drafts[s, j] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), V - 1)
            else:            # a drafter certain of its token: often the target's likeliest one
                drafts[s, j] = int(np.argmax(logits[s, j])) if rng.random() < 0.7 else int(rng.integers(0, V))
    ua = rng.random((n, K)).astype(np.float32)
    us = rng.random((n, K + 1)).astype(np.float32)
    return logits, drafts, q, ua, us


@pytest.mark.parametrize("V,n,with_q,temp", [(1000, 48, False, 1.0), (1000, 48, True, 0.7), (129280, 6, False, 1.0),
                                             (129280, 4, True, 1.3)])
def test_parity_with_oracle(V, n, with_q, temp):
    rng = np.random.default_rng(V + n + int(with_q))
    K = 3
    logits, drafts, q, ua, us = _inputs(rng, n, K, V, with_q)
    acc, tok = _run(logits, drafts, q, ua, us, temp)
    exempt = 0
    for s in range(n):
        tr = {}
        a, t = smp.rejection_sample(logits[s].astype(np.float64), drafts[s], None if q is None else q[s],
                                    ua[s].astype(np.float64), us[s].astype(np.float64), temp, tr)
        if (int(acc[s]), int(tok[s])) == (a, t):
            continue
        m = tr["accept_margins"]
        near = min(m[: min(a, int(acc[s])) + 1]) < TIE if m else False
        near = near or (int(acc[s]) == a and tr["sample_margin"] < TIE)
        assert near, f"sequence {s}: GPU {(int(acc[s]), int(tok[s]))} vs oracle {(a, t)} away from any threshold"
        exempt += 1
    assert exempt * 10 <= n, f"{exempt} of {n} sequences decided within {TIE} of a threshold"
    assert ((acc >= 0) & (acc <= K) & (tok >= 0) & (tok < V)).all()


def test_emitted_tokens_follow_the_target():
    rng = np.random.default_rng(21)
    n, K, V = 200_000, 2, 16
    base = rng.standard_normal((K + 1, V)) * 1.2
    q1 = rng.dirichlet(np.ones(V) * 0.8, size=K)
    logits = np.broadcast_to(base, (n, K + 1, V)).copy()
    q = np.broadcast_to(q1, (n, K, V)).copy()
    drafts = np.stack([rng.choice(V, size=n, p=q1[j]) for j in range(K)], axis=1)
    ua = rng.random((n, K))
    us = rng.random((n, K + 1))
    acc, tok = _run(logits, drafts, q, ua, us, 1.0)
    assert ((acc >= 0) & (acc <= K)).all()
    first = np.where(acc >= 1, drafts[:, 0], tok)
    second = np.where(acc >= 2, drafts[:, 1], tok)[acc >= 1]
    for emitted, p in ((first, smp.target_probs(base[0], 1.0)), (second, smp.target_probs(base[1], 1.0))):
        obs = np.bincount(emitted, minlength=V).astype(np.float64)
        exp = p * len(emitted)
        chi2 = float(((obs - exp) ** 2 / exp).sum())
        assert chi2 < 60.0, f"chi-square {chi2:.1f} with {V - 1} degrees of freedom"
    # and the drafter's own law is far from the target's: the test can fail
    obs = np.bincount(drafts[:, 0], minlength=V).astype(np.float64)
    exp = smp.target_probs(base[0], 1.0) * n
    assert float(((obs - exp) ** 2 / exp).sum()) > 1000.0


def test_greedy_limit_is_the_greedy_rule():
    rng = np.random.default_rng(22)
    n, K, V = 64, 5, 4096
    g = rng.integers(0, V, (n, K + 1))
    logits = rng.standard_normal((n, K + 1, V)).astype(np.float32)
    for s in range(n):
        logits[s, np.arange(K + 1), g[s]] += 60.0
    drafts = np.where(rng.random((n, K)) < 0.7, g[:, :K], rng.integers(0, V, (n, K)))
    acc, tok = _run(logits, drafts, None, rng.random((n, K)), rng.random((n, K + 1)), 0.05)
    for s in range(n):
        assert (int(acc[s]), int(tok[s])) == oracle.accept(list(drafts[s]), list(g[s]))


def test_errors_are_reported():
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(23)
    logits, drafts, _, ua, us = _inputs(rng, 3, 2, 64, False)
    drafts[1, 0] = 64                                   # not a token
    acc, tok = _run(logits, drafts, None, ua, us, 1.0)
    assert (int(acc[1]), int(tok[1])) == (-1, -1)
    assert acc[0] >= 0 and acc[2] >= 0
    with pytest.raises(B.SpecError):
        _run(logits[:, :, :62], drafts, None, ua, us, 1.0)     # vocab not a multiple of 4
    with pytest.raises(B.SpecError):
        _run(logits, drafts, None, ua, us, 0.0)                 # temperature must be positive
