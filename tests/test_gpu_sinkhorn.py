"""Sinkhorn normalisation (training-time token-group balance, gist.science/nl
Kerncomponenten 2; gist.science/zh technical summary 2.1.1) against the
oracle: P, log u and log v element by element on seeded affinities, from one
round to convergence, K from 1 to 1000, and the n = 1M, K = 256 shape.

Tolerance, from the arithmetic: the kernel works in fp32 with base-2
log-sum-exp per token and fp32 sums of at most a few hundred row-normalised
entries per warp before the per-column sum of the CTAs' partials; each
potential is the log of a sum of positive terms (no cancellation), so its
error is a few float ulps of the sum, a few 1e-7 relative per round.  P is
exp of (S / tau + log u + log v), whose exponent carries about |S| / tau
times 1e-7 of rounding.  Bound used: |d log u|, |d log v| <= 2e-5 * rounds
(at least 1e-5) + 1e-6 * max |S| / tau, and |dP| <= 1e-6 + that bound * P."""
import numpy as np
import pytest
import torch

import oracle
import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    yield
    torch.cuda.empty_cache()


def _bound(S, tau, iters):
    return max(1e-5, 2e-5 * iters) + 1e-6 * float(np.abs(S).max()) / tau


def _check(S_np, tau, iters, P, lu, lv, rows=None, label=""):
    Pr, lur, lvr = oracle.sinkhorn(S_np, tau, iters, want_p=rows is None)
    tol = _bound(S_np, tau, iters)
    du = np.abs(lu.cpu().numpy() - lur).max()
    dv = np.abs(lv.cpu().numpy() - lvr).max()
    assert du <= tol and dv <= tol, f"{label}: log u {du:.3e}, log v {dv:.3e}, bound {tol:.3e}"
    if P is None:
        return
    if rows is None:
        Pg, Pref = P.cpu().numpy(), Pr
    else:
        b, i = rows // S_np.shape[1], rows % S_np.shape[1]
        Pg = P[torch.as_tensor(b), torch.as_tensor(i)].cpu().numpy()
        Pref = np.exp(S_np[b, i].astype(np.float64) / tau + lur[b, i][:, None] + lvr[b][:, :])
    err = np.abs(Pg - Pref) - (1e-6 + tol * np.abs(Pref))
    assert np.isfinite(Pg).all(), f"{label}: non-finite P"
    assert err.max() <= 0, f"{label}: P off by {np.abs(Pg - Pref).max():.3e}"


CASES = [
    # B, n, K, tau, iters
    (1, 100, 8, 1.0, 1),
    (2, 1000, 64, 0.5, 3),
    (1, 5000, 256, 1.0, 10),
    (3, 77, 1000, 2.0, 2),      # K not a multiple of 32, the largest lane count
    (1, 1, 5, 1.0, 3),          # one token
    (2, 333, 1, 1.0, 2),        # one group: P = 1
    (1, 2000, 33, 1.0, 60),     # converged: token masses 1 as well
    (400, 20, 16, 1.0, 4),      # more sequences than CTAs per sequence
    (2, 50000, 33, 0.7, 3),     # the plain-load sweep over many rows
    (3, 4099, 100, 1.0, 5),     # the bulk sweep with four lanes per row and a ragged last chunk
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}n{}K{}t{}r{}".format(*c))
def test_sinkhorn_matches_oracle(case):
    B, n, K, tau, iters = case
    g = torch.Generator(device="cuda").manual_seed(n * 7 + K)
    S = (2.0 * torch.randn(B, n, K, generator=g, device="cuda")).contiguous()
    P, lu, lv = fg.focus_sinkhorn(S, tau, iters)
    torch.cuda.synchronize()
    S_np = S.cpu().numpy()
    _check(S_np, tau, iters, P, lu, lv, label=str(case))
    cols = P.sum(dim=1).cpu().numpy()
    np.testing.assert_allclose(cols, n / K, rtol=1e-4)
    if iters >= 60:
        np.testing.assert_allclose(P.sum(dim=2).cpu().numpy(), 1.0, rtol=1e-4)
    # potentials only
    P2, lu2, lv2 = fg.focus_sinkhorn(S, tau, iters, want_p=False)
    assert P2 is None
    assert torch.equal(lu2, lu) and torch.equal(lv2, lv)


def test_sinkhorn_at_one_million_tokens():
    """The n = 1M workload's shape (K = 256) on affinities with the mixture's
    structure, 3 rounds: every potential, and P on 4096 seeded rows."""
    w = synth.workload(4)
    comp = synth.make_components(w, "cuda")
    S = synth.synthetic_affinities(w, comp, device="cuda")
    P, lu, lv = fg.focus_sinkhorn(S, 1.0, 3)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(0).choice(w.n, 4096, replace=False)).astype(np.int64)
    _check(S.cpu().numpy(), 1.0, 3, P, lu, lv, rows=rows, label="n1m")
    np.testing.assert_allclose(P.sum(dim=1).cpu().numpy(), w.n / w.K, rtol=1e-4)
    del P, S
    torch.cuda.empty_cache()
