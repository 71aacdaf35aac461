"""Rejection-sampling verification on the GPU against the oracle
(oracle/sampling.py) and against the law it must produce, through both entry
points: spec_rejection_sample (one block per sequence) and
spec_rejection_sample_ws (row statistics split over many blocks).

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


@pytest.fixture(params=["block", "split"])
def form(request):
    return request.param


def _run(logits, drafts, q, ua, us, temperature, form="block", ws=None):
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    n, K1, V = logits.shape
    acc = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    args = (_dev(logits.astype(np.float32)), _dev(drafts.astype(np.int32)) if K1 > 1 else None,
            None if q is None else _dev(q.astype(np.float32)),
            _dev(ua.astype(np.float32)) if K1 > 1 else None, _dev(us.astype(np.float32)),
            n, K1 - 1, V, temperature, acc, tok)
    if form == "block":
        B.spec_rejection_sample(*args, 0)
    else:
        nb = B.spec_rejection_sample_ws_bytes(n, K1 - 1)
        if ws is None:
            ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        B.spec_rejection_sample_ws(*args, ws, nb, 0)
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
def test_parity_with_oracle(V, n, with_q, temp, form):
    rng = np.random.default_rng(V + n + int(with_q))
    K = 3
    logits, drafts, q, ua, us = _inputs(rng, n, K, V, with_q)
    acc, tok = _run(logits, drafts, q, ua, us, temp, form)
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


def test_emitted_tokens_follow_the_target(form):
    rng = np.random.default_rng(21)
    n, K, V = 200_000, 2, 16
    base = rng.standard_normal((K + 1, V)) * 1.2
    q1 = rng.dirichlet(np.ones(V) * 0.8, size=K)
    logits = np.broadcast_to(base, (n, K + 1, V)).copy()
    q = np.broadcast_to(q1, (n, K, V)).copy()
    drafts = np.stack([rng.choice(V, size=n, p=q1[j]) for j in range(K)], axis=1)
    ua = rng.random((n, K))
    us = rng.random((n, K + 1))
    acc, tok = _run(logits, drafts, q, ua, us, 1.0, form)
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


@pytest.mark.parametrize("n,V", [(64, 4096), (12, 129280)])
def test_greedy_limit_is_the_greedy_rule(form, n, V):
    rng = np.random.default_rng(22)
    K = 5
    g = rng.integers(0, V, (n, K + 1))
    logits = rng.standard_normal((n, K + 1, V)).astype(np.float32)
    for s in range(n):
        logits[s, np.arange(K + 1), g[s]] += 60.0
    drafts = np.where(rng.random((n, K)) < 0.7, g[:, :K], rng.integers(0, V, (n, K)))
    acc, tok = _run(logits, drafts, None, rng.random((n, K)), rng.random((n, K + 1)), 0.05, form)
    for s in range(n):
        assert (int(acc[s]), int(tok[s])) == oracle.accept(list(drafts[s]), list(g[s]))


def test_errors_are_reported(form):
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(23)
    logits, drafts, _, ua, us = _inputs(rng, 3, 2, 64, False)
    drafts[1, 0] = 64                                   # not a token
    acc, tok = _run(logits, drafts, None, ua, us, 1.0, form)
    assert (int(acc[1]), int(tok[1])) == (-1, -1)
    assert acc[0] >= 0 and acc[2] >= 0
    with pytest.raises(B.SpecError):
        _run(logits[:, :, :62], drafts, None, ua, us, 1.0, form)     # vocab not a multiple of 4
    with pytest.raises(B.SpecError):
        _run(logits, drafts, None, ua, us, 0.0, form)                 # temperature must be positive


def test_split_form_workspace_is_checked():
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(24)
    logits, drafts, _, ua, us = _inputs(rng, 4, 3, 256, False)
    nb = B.spec_rejection_sample_ws_bytes(4, 3)
    assert nb >= 4 * 4 * min(64, -(-1024 // 16)) * 8        # at least the rows' partial statistics
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    acc = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(B.SpecError) as e:
        B.spec_rejection_sample_ws(_dev(logits), _dev(drafts.astype(np.int32)), None, _dev(ua), _dev(us), 4, 3, 256,
                                   1.0, acc, acc, ws, nb - 8, 0)
    assert e.value.code == B.SPEC_ERR_ARG


def test_split_form_workspace_is_reusable():
    """Each call leaves its counters at zero: calls in a row on one workspace
    give what calls on fresh workspaces give (rows walked by several blocks
    per sequence, with and without a drafter distribution)."""
    import torch
    from lossless_speculative_decoding_gb300 import binding as B
    rng = np.random.default_rng(25)
    n, K, V = 8, 3, 129280
    nb = B.spec_rejection_sample_ws_bytes(n, K)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    for with_q in (False, True, False):
        logits, drafts, q, ua, us = _inputs(rng, n, K, V, with_q)
        got = _run(logits, drafts, q, ua, us, 1.0, "split", ws=ws)
        fresh = _run(logits, drafts, q, ua, us, 1.0, "split")
        assert (got[0] == fresh[0]).all() and (got[1] == fresh[1]).all()
        assert int(ws[: 8 * n].sum().item()) == 0, "counters left non-zero"
