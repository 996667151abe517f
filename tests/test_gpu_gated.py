"""Soft-gated attention of training (gist.science/zh technical summary 2.1.2;
gist.science/nl Kerncomponent 4) and its backward against the oracle: O and
the log-sum-exp, then dQ, dK, dV, dG and d lambda, element by element, on
seeded inputs with ragged tails, GQA, both head sizes, K_g from 5 to 128,
window 0, a window wider than the sequence and a negative lambda.

Tolerances, from the arithmetic: the forward rounds P to bf16 for P V (as the
inference path does), so O is held to the inference bar (max-abs 1e-2,
mean-abs 1e-3, log-sum-exp 2e-3).  The backward's products take P, dS and dt
in bf16 (relative rounding 2^-9) and da in fp16 (2^-12), against fp32 sums
of up to n terms of both signs; each gradient is held to a max-abs error of
1e-2 and a mean-abs error of 5e-4, both relative to the largest magnitude of
that gradient (measured: at most 3.9e-3 and 1.2e-4 on these cases), and
d lambda, a sum over all gated pairs of terms of both signs, to 2^-8 of the
sum of the terms' magnitudes (the condition of that sum: the result itself
can be far smaller than its terms) or 1e-2 of the result if larger."""
import numpy as np
import pytest
import torch

import oracle
import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build, synth
from _gpu_helpers import check_output

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    yield
    torch.cuda.empty_cache()


def _inputs(B, n, Hq, Hkv, d, Kg, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    Q = torch.randn(B, n, Hq, d, generator=g, device="cuda").to(torch.bfloat16)
    K = torch.randn(B, n, Hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn(B, n, Hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    G = torch.softmax(2.0 * torch.randn(B, n, Kg, generator=g, device="cuda"), dim=-1)
    dO = torch.randn(B, n, Hq, d, generator=g, device="cuda").to(torch.bfloat16)
    return Q, K, V, G.contiguous(), dO


def _close(name, got, ref, max_rel=1e-2, mean_rel=5e-4):
    got = got.detach().float().cpu().numpy().reshape(ref.shape)
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{name}: non-finite"
    assert err.max() <= max_rel * scale and err.mean() <= mean_rel * scale, (
        f"{name}: max {err.max():.3e} mean {err.mean():.3e} scale {scale:.3e}")


CASES = [
    # B, n, Hq, Hkv, d, Kg, window, lambda
    (1, 200, 2, 2, 64, 16, 32, 4.0),
    (2, 130, 4, 1, 128, 64, 0, 2.0),
    (1, 64, 2, 2, 64, 5, 10 ** 6, 3.0),
    (1, 300, 8, 2, 128, 128, 64, -1.5),
    (1, 1, 2, 1, 64, 16, 4, 1.0),
    (2, 257, 4, 4, 128, 33, 1, 6.0),
    (1, 700, 4, 2, 64, 16, 200, 2.5),   # tiles wholly inside, across and outside the window
    (2, 150, 16, 2, 64, 48, 8, 3.0),    # GQA 8:1, two head chunks for dG
    (1, 390, 3, 1, 128, 64, 100, 2.0),  # GQA 3:1 (odd: consecutive query tiles share a CTA)
    (2, 1100, 4, 2, 128, 64, 128, 2.5), # d 128, K_g 64 as in training: the streams wrap their
                                        # stage rings many times, two heads per key-side CTA
    (1, 260, 4, 4, 64, 100, 40, 2.0),   # d 64 with K_g > 64: the key side keeps P and dT over
                                        # the A product's TMEM columns
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}n{}H{}x{}d{}Kg{}w{}l{}".format(*c))
def test_gated_fwd_bwd_match_oracle(case):
    B, n, Hq, Hkv, d, Kg, window, lam = case
    Q, K, V, G, dO = _inputs(B, n, Hq, Hkv, d, Kg, seed=n + Kg)
    O, lse = fg.focus_gated_attention_fwd(Q, K, V, G, window, lam)
    dQ, dK, dV, dG, dl = fg.focus_gated_attention_bwd(Q, K, V, G, O, lse, dO, window, lam)
    torch.cuda.synchronize()
    Qb, Kb, Vb = synth.bits(Q), synth.bits(K), synth.bits(V)
    Gn = G.cpu().numpy()
    Oref, Lref = oracle.gated_fwd(Qb, Kb, Vb, Gn, window, lam)
    check_output(O, Oref.astype(np.float32), lse, Lref.astype(np.float32), label=str(case))
    # the backward from the GPU's own O (its dO . O term), in double
    ref = oracle.gated_bwd(Qb, Kb, Vb, Gn, dO.float().cpu().numpy(), window, lam, with_abs=True)
    for name, got, r in zip(("dQ", "dK", "dV", "dG"), (dQ, dK, dV, dG), ref[:4]):
        _close(f"{case} {name}", got, r)
    dl_ref, dl_abs = ref[4], ref[5]
    # a sum of per-pair terms of both signs: judged against the sum of their
    # magnitudes at 2^-8 (each term carries the bf16 rounding of O through
    # D_i and of the gate's operands), or 1e-2 of the result when that is larger
    tol = max(1e-2 * abs(dl_ref), 2.0 ** -8 * dl_abs, 1e-9)
    assert abs(float(dl) - dl_ref) <= tol, (float(dl), dl_ref, dl_abs)
    # deterministic: a second run repeats every bit
    again = fg.focus_gated_attention_bwd(Q, K, V, G, O, lse, dO, window, lam)
    for x, y in zip((dQ, dK, dV, dG, dl), again):
        assert torch.equal(x, y)


def test_gated_fwd_many_items_per_cta():
    """More work items than SMs (192 pairs of 128-row query tiles), so every
    CTA of the persistent forward walks several items through its barrier
    phases; a ragged last tile; every output row against the oracle."""
    B, n, Hq, Hkv, d, Kg, window, lam = 1, 3000, 16, 16, 128, 64, 256, 3.0
    Q, K, V, G, _ = _inputs(B, n, Hq, Hkv, d, Kg, seed=11)
    O, lse = fg.focus_gated_attention_fwd(Q, K, V, G, window, lam)
    torch.cuda.synchronize()
    Oref, Lref = oracle.gated_fwd(synth.bits(Q), synth.bits(K), synth.bits(V), G.cpu().numpy(),
                                  window, lam)
    check_output(O, Oref.astype(np.float32), lse, Lref.astype(np.float32), label="n3000 H16")
