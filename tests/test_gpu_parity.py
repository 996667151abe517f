"""GPU parity: every CUDA entry point against the CPU oracle, element by
element, on seeded inputs that span several 128-row tiles, ragged tails and
the degenerate cases of the method (window 0, window >= n, one group holding
every token, top-k = K, n = 1, K = 1024 with top-8, GQA ratios 1/4/8)."""
import numpy as np
import pytest
import torch

import oracle
import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build, synth
from _gpu_helpers import check_ids, check_output, free_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    fg.focus_get_device_status(reset=True)
    yield
    assert fg.focus_get_device_status(reset=True) == 0, "a device-side wait timed out"
    free_cuda()


def rand_ids(B, n, K, topk, seed, zipf=0.0):
    rng = np.random.default_rng(seed)
    p = np.arange(1, K + 1, dtype=np.float64) ** (-zipf) if zipf else np.ones(K)
    p /= p.sum()
    ids = np.empty((B, n, topk), np.int32)
    for b in range(B):
        for i in range(n):
            ids[b, i] = rng.choice(K, size=topk, replace=False, p=p)
    return ids


def qkv(B, n, Hq, Hkv, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    Q = torch.randn(B, n, Hq, d, generator=g, device="cuda", dtype=torch.bfloat16)
    K = torch.randn(B, n, Hkv, d, generator=g, device="cuda", dtype=torch.bfloat16)
    V = torch.randn(B, n, Hkv, d, generator=g, device="cuda", dtype=torch.bfloat16)
    return Q, K, V


ATTN_CASES = [
    # B, n, Hq, Hkv, d, K, topk, window
    (1, 300, 2, 2, 64, 4, 1, 16),
    (1, 1000, 4, 1, 128, 8, 2, 64),
    (2, 777, 8, 1, 128, 5, 3, 200),
    (1, 513, 2, 2, 64, 16, 1, 0),
    (1, 400, 2, 2, 128, 3, 3, 1),
    (1, 640, 2, 2, 64, 1, 1, 32),
    (1, 333, 2, 1, 128, 100, 4, 2000),
    (1, 900, 2, 2, 128, 128, 4, 128),
    (1, 1, 2, 2, 64, 4, 2, 16),
    (1, 129, 2, 2, 64, 1024, 8, 7),
    (2, 1500, 4, 2, 128, 64, 2, 256),
    (1, 1100, 6, 2, 128, 16, 2, 100),     # odd GQA ratio: query tiles pair up
    (1, 2300, 3, 3, 64, 12, 3, 300),      # odd number of query tiles per head
    (1, 600, 2, 2, 128, 1024, 8, 96),     # the largest K and topk at d = 128
    (4, 300, 2, 2, 64, 1024, 2, 16),      # B * K at its limit (4096), most groups empty
    (1, 1500, 2, 2, 128, 4, 2, 700),      # a row's window holds ~350 members of its groups:
                                          # the group kernel's window bound spans key tiles
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: "B{}n{}H{}x{}d{}K{}k{}w{}".format(*c))
def test_attention_matches_oracle(case):
    B, n, Hq, Hkv, d, K, topk, window = case
    Q, Kt, V = qkv(B, n, Hq, Hkv, d, seed=n + K)
    ids_np = rand_ids(B, n, K, topk, seed=7 * n + K)
    ids = torch.from_numpy(ids_np).cuda()
    off, pos, inv = fg.focus_bucket(ids, K)
    O, L = fg.focus_attention_fwd(Q, Kt, V, window, ids, off, pos, inv, K)
    torch.cuda.synchronize()
    Oref, Lref = oracle.attention(synth.bits(Q), synth.bits(Kt), synth.bits(V), ids_np, window)
    check_output(O, Oref, L.permute(0, 2, 1), Lref, label=str(case))


@pytest.mark.parametrize("B,n,Hq,Hkv,d", [(1, 300, 2, 2, 64), (2, 1000, 8, 2, 128),
                                         (1, 129, 1, 1, 128), (1, 2048, 4, 4, 64),
                                         (1, 700, 3, 1, 128)])
def test_dense_causal_matches_oracle(B, n, Hq, Hkv, d):
    Q, Kt, V = qkv(B, n, Hq, Hkv, d, seed=3 * n)
    O, L = fg.focus_dense_causal_fwd(Q, Kt, V, with_lse=True)
    torch.cuda.synchronize()
    ids0 = np.zeros((B, n, 1), np.int32)
    Oref, Lref = oracle.attention(synth.bits(Q), synth.bits(Kt), synth.bits(V), ids0, n)
    check_output(O, Oref, L.permute(0, 2, 1), Lref, label="dense")


@pytest.mark.parametrize("B,n,Hq,Hkv,d,K,topk,window", [
    (1, 1000, 4, 2, 128, 1, 1, 64),     # one group holds every token
    (2, 777, 4, 1, 64, 8, 2, 5000),     # the window covers every causal pair
    (1, 1300, 6, 2, 128, 4, 4, 0),      # topk = K: every pair is scored in group 0
])
def test_special_cases_reduce_to_dense_causal(B, n, Hq, Hkv, d, K, topk, window):
    """Where the allowed set is every causal pair, the Focus path (group,
    window and merge kernels) must give plain causal attention: checked
    against the library's own dense kernel, an independent mainloop run.
    Each output is within (1e-2 max-abs, 1e-3 mean-abs) of the exact result
    (the oracle tests), so the two agree within twice that; each is rounded
    to bf16 on its own, and one bf16 step at |O| in [2, 4) is already
    1.6e-2."""
    Q, Kt, V = qkv(B, n, Hq, Hkv, d, seed=5 * n + K)
    ids = torch.from_numpy(rand_ids(B, n, K, topk, seed=n + 3 * K)).cuda()
    off, pos, inv = fg.focus_bucket(ids, K)
    O, L = fg.focus_attention_fwd(Q, Kt, V, window, ids, off, pos, inv, K)
    Od, Ld = fg.focus_dense_causal_fwd(Q, Kt, V, with_lse=True)
    torch.cuda.synchronize()
    err = (O.float() - Od.float()).abs()
    assert torch.isfinite(O.float()).all()
    assert float(err.max()) <= 2e-2 and float(err.mean()) <= 2e-3, \
        f"K{K} top{topk} w{window}: max-abs {float(err.max()):.3e} mean-abs {float(err.mean()):.3e}"
    assert float((L - Ld).abs().max()) <= 2 * 2e-3   # twice the lse bound


@pytest.mark.parametrize("B,n,K,topk", [(1, 1, 4, 2), (2, 5000, 64, 2), (3, 4097, 7, 3),
                                        (1, 3000, 1024, 8), (1, 9000, 1, 1), (2, 20000, 256, 2)])
def test_bucket_matches_oracle_exactly(B, n, K, topk):
    ids_np = rand_ids(B, n, K, topk, seed=n + K, zipf=1.1 if K > 8 else 0.0)
    off, pos, inv = fg.focus_bucket(torch.from_numpy(ids_np).cuda(), K)
    roff, rpos, rinv = oracle.bucket(ids_np, K)
    np.testing.assert_array_equal(off.cpu().numpy(), roff)
    np.testing.assert_array_equal(pos.cpu().numpy(), rpos)
    np.testing.assert_array_equal(inv.cpu().numpy(), rinv)


@pytest.mark.parametrize("w", [synth.small(B=2, n=500, hidden=256, dg=64, K=32, topk=3,
                                           x_kind="normal", seed=11),
                               synth.small(n=700, hidden=4096, dg=128, K=256, topk=2, seed=12),
                               synth.small(n=300, hidden=512, dg=200, K=40, topk=4, seed=13),
                               synth.small(n=200, hidden=128, dg=16, K=1000, topk=8,
                                           x_kind="normal", seed=14),
                               synth.small(n=100, hidden=64, dg=32, K=1, topk=1, seed=15),
                               # more centroids than centroid dimensions: (X W_g) C^T
                               synth.small(B=2, n=1000, hidden=1024, dg=64, K=100, topk=4,
                                           seed=16),
                               synth.small(n=333, hidden=192, dg=20, K=80, topk=3,
                                           x_kind="normal", seed=17),
                               synth.small(n=513, hidden=640, dg=128, K=144, topk=8, seed=18),
                               synth.small(n=1, hidden=256, dg=64, K=128, topk=2, seed=19)],
                         ids=lambda w: w.label)
def test_assign_matches_oracle(w):
    Wg, C = synth.make_params(w, "cuda")
    comp = synth.make_components(w, "cuda")
    X = synth.make_x(w, Wg, C, comp, "cuda")
    ids, margin = fg.focus_assign(X, Wg, C, w.topk)
    torch.cuda.synchronize()
    rids, rmargin, _ = oracle.assign(synth.bits(X), Wg.cpu().numpy(), C.cpu().numpy(), w.topk)
    skipped = check_ids(ids, rids, rmargin)
    # near-ties (margin <= 1e-4) are ambiguous and skipped; they must stay rare
    assert skipped <= max(8, w.B * w.n // 50), skipped
    sure = rmargin > 1e-4
    np.testing.assert_allclose(margin.cpu().numpy()[sure], rmargin[sure], atol=5e-5, rtol=1e-4)


# (the window kernel takes every pair with i - j < w, the group kernel the
# shared pairs further back: w = 300 with 6 groups over 700 tokens puts about
# a hundred members of each group inside a row's window, so the group
# kernel's window bound masks whole key tiles; w > n leaves it nothing)
@pytest.mark.parametrize("case", [(1, 700, 6, 2, 40), (2, 1000, 64, 2, 256), (1, 600, 128, 4, 16),
                                  (1, 300, 5, 5, 3), (1, 260, 9, 1, 0), (1, 700, 6, 2, 300),
                                  (2, 900, 3, 2, 1000)])
def test_every_allowed_pair_scored_exactly_once(case):
    B, n, K, topk, window = case
    ids_np = rand_ids(B, n, K, topk, seed=n * 3 + K)
    ids = torch.from_numpy(ids_np).cuda()
    off, pos, inv = fg.focus_bucket(ids, K)
    Q, Kt, V = qkv(B, n, 2, 2, 64, seed=5)
    _, _, cnt = fg.focus_attention_fwd_counted(Q, Kt, V, window, ids, off, pos, inv, K)
    per, tot = fg.focus_count_pairs(ids, off, pos, inv, K, window)
    torch.cuda.synchronize()
    rper, rtot = oracle.count_pairs(ids_np, window)
    np.testing.assert_array_equal(cnt.cpu().numpy(), rper)
    np.testing.assert_array_equal(per.cpu().numpy(), rper)
    _, share = oracle.count_pairs(ids_np, 0)
    assert tot.cpu().tolist() == [rtot, share]


def test_deterministic_and_prefill_paths_agree():
    w = synth.small(B=2, n=1100, hidden=512, Hq=4, Hkv=2, d=128, K=16, dg=64, topk=2,
                    window=100, seed=21)
    t = synth.make_all(w, "cuda")
    ids, _ = fg.focus_assign(t["X"], t["Wg"], t["C"], w.topk)
    off, pos, inv = fg.focus_bucket(ids, w.K)
    O1, L1 = fg.focus_attention_fwd(t["Q"], t["K"], t["V"], w.window, ids, off, pos, inv, w.K)
    O2, L2 = fg.focus_attention_fwd(t["Q"], t["K"], t["V"], w.window, ids, off, pos, inv, w.K)
    ids_out = torch.empty_like(ids)
    L3 = torch.empty_like(L1)
    O3, _ = fg.focus_prefill(t["X"], t["Wg"], t["C"], t["Q"], t["K"], t["V"], w.topk, w.window,
                             lse=L3, ids_out=ids_out)
    host = {k: t[k].cpu().pin_memory() for k in ("X", "Wg", "C", "Q", "K", "V")}
    L4 = torch.empty(L1.shape, dtype=torch.float32).pin_memory()
    O4, _ = fg.focus_prefill(host["X"], host["Wg"], host["C"], host["Q"], host["K"], host["V"],
                             w.topk, w.window, lse=L4)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    assert torch.equal(ids_out, ids)
    assert torch.equal(O3, O1) and torch.equal(L3, L1)
    assert torch.equal(O4, O1.cpu()) and torch.equal(L4, L1.cpu())
    assert fg.focus_last_launch_count() >= 8
