"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: a worked example
derived by hand, brute-force enumeration of the allowed-pair rule with
Python sets, special cases that reduce to a library routine
(torch scaled_dot_product_attention in float64 with a causal, band or
explicit mask; numpy stable argsort; numpy bincount/cumsum), and closed
forms for the pair counts.  Each case is chosen so that a plausible slip in
the oracle (window off by one, dropped causality, wrong GQA head map, wrong
scale, transposed projection, wrong tie-break) fails at least one test.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from learned_group_sparse_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers ---

def _bf16_bits(x):
    return synth.bits(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def _rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _brute_allowed(ids, window):
    """Boolean [B, n, n] allowed-pair matrix by enumeration with Python sets."""
    B, n, _ = ids.shape
    A = np.zeros((B, n, n), dtype=bool)
    for b in range(B):
        sets = [set(int(g) for g in ids[b, i]) for i in range(n)]
        for i in range(n):
            for j in range(i + 1):
                A[b, i, j] = (i - j < window) or bool(sets[i] & sets[j])
    return A


def _sdpa(Q, K, V, mask=None, causal=False):
    """torch SDPA in float64 on [B, n, H, d] bf16 inputs (GQA by repeat)."""
    q = Q.double().permute(0, 2, 1, 3)
    k = K.double().permute(0, 2, 1, 3)
    v = V.double().permute(0, 2, 1, 3)
    rep = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(rep, dim=1)
    v = v.repeat_interleave(rep, dim=1)
    m = None if mask is None else torch.as_tensor(mask)[:, None, :, :]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, is_causal=causal)
    return o.permute(0, 2, 1, 3).numpy()


def _lse(Q, K, mask):
    q = Q.double().permute(0, 2, 1, 3)
    k = K.double().permute(0, 2, 1, 3)
    k = k.repeat_interleave(q.shape[1] // k.shape[1], dim=1)
    s = (q @ k.transpose(-1, -2)) / np.sqrt(q.shape[-1])
    s = s.masked_fill(~torch.as_tensor(mask)[:, None], float("-inf"))
    return torch.logsumexp(s, dim=-1).permute(0, 2, 1).numpy()


def _qkv(B, n, Hq, Hkv, d, seed):
    return (_rand_bf16((B, n, Hq, d), seed), _rand_bf16((B, n, Hkv, d), seed + 1),
            _rand_bf16((B, n, Hkv, d), seed + 2))


def _run(Q, K, V, ids, window, rows=None):
    return oracle.attention(synth.bits(Q), synth.bits(K), synth.bits(V), ids, window, rows=rows)


def _rand_ids(B, n, K, topk, seed):
    rng = np.random.default_rng(seed)
    ids = np.empty((B, n, topk), np.int32)
    for b in range(B):
        for i in range(n):
            ids[b, i] = rng.choice(K, size=topk, replace=False)
    return ids


# ------------------------------------------------------------ hand example ---

def test_hand_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "hand_worked_example.json")))
    n, d = ex["n"], ex["d"]
    ids = np.array(ex["ids"], np.int32).reshape(1, n, 1)
    Q = torch.zeros(1, n, 1, d, dtype=torch.bfloat16)
    K = _rand_bf16((1, n, 1, d), 3)                 # irrelevant when Q = 0
    V = torch.tensor(ex["V"], dtype=torch.float32).view(1, n, 1, d).to(torch.bfloat16)
    O, L = _run(Q, K, V, ids, ex["window"])
    np.testing.assert_allclose(O[0, :, 0], np.array(ex["O"]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(L[0, :, 0], np.log(np.array(ex["count"], float)), atol=1e-6)
    per, tot = oracle.count_pairs(ids, ex["window"])
    assert per[0].tolist() == ex["count"] and tot == sum(ex["count"])
    A = _brute_allowed(ids, ex["window"])[0]
    assert [list(np.nonzero(A[i])[0]) for i in range(n)] == ex["allowed"]


# -------------------------------------------------------------- mask pins ---

@pytest.mark.parametrize("n,K,topk,window,seed", [
    (40, 6, 2, 5, 0), (37, 3, 1, 1, 1), (33, 9, 3, 0, 2), (48, 5, 2, 7, 3), (20, 4, 4, 3, 4)])
def test_mask_by_one_hot_values(n, K, topk, window, seed):
    """Q = 0 and V[j] = e_j expose the allowed set: O[i, j] = 1/|A_i| on it."""
    B = 2
    ids = _rand_ids(B, n, K, topk, seed)
    d = 64
    Q = torch.zeros(B, n, 1, d, dtype=torch.bfloat16)
    Kt = _rand_bf16((B, n, 1, d), seed)
    V = torch.zeros(B, n, 1, d)
    for j in range(n):
        V[:, j, 0, j] = 1.0
    O, _ = _run(Q, Kt, V.to(torch.bfloat16), ids, window)
    A = _brute_allowed(ids, window)
    expect = A / A.sum(-1, keepdims=True)
    np.testing.assert_allclose(O[:, :, 0, :n], expect, atol=1e-6)
    per, tot = oracle.count_pairs(ids, window)
    assert (per == A.sum(-1)).all() and tot == int(A.sum())


# ------------------------------------------ reductions to library routines ---

@pytest.mark.parametrize("case", ["one_group", "topk_eq_K", "window_ge_n"])
def test_reduces_to_dense_causal(case):
    B, n, Hq, Hkv, d = 2, 70, 4, 2, 32
    Q, K, V = _qkv(B, n, Hq, Hkv, d, 11)
    if case == "one_group":
        ids, window = np.zeros((B, n, 1), np.int32), 3
    elif case == "topk_eq_K":
        ids, window = _rand_ids(B, n, 3, 3, 5), 2
    else:
        ids, window = _rand_ids(B, n, 16, 1, 6), n
    O, L = _run(Q, K, V, ids, window)
    ref = _sdpa(Q, K, V, causal=True)
    np.testing.assert_allclose(O, ref, atol=2e-6)
    causal = np.tril(np.ones((n, n), bool))[None].repeat(B, 0)
    np.testing.assert_allclose(L, _lse(Q, K, causal), atol=2e-5)


@pytest.mark.parametrize("window", [1, 4, 9])
def test_disjoint_groups_reduce_to_sliding_window(window):
    B, n, H, d = 1, 64, 3, 16
    Q, K, V = _qkv(B, n, H, H, d, 21)
    ids = np.arange(n, dtype=np.int32).reshape(1, n, 1)      # K = n, nobody shares
    O, _ = _run(Q, K, V, ids, window)
    band = torch.ones(n, n).tril().bool() & ~torch.ones(n, n).tril(-window).bool()
    ref = _sdpa(Q, K, V, mask=band[None])
    np.testing.assert_allclose(O, ref, atol=2e-6)


@pytest.mark.parametrize("window", [0, 1])
def test_no_window_reduces_to_per_group_causal(window):
    """With no window and top-1 groups, each group is plain causal attention
    over its own gathered rows."""
    B, n, H, d, K = 1, 90, 2, 32, 4
    Q, Kt, V = _qkv(B, n, H, H, d, 31)
    ids = _rand_ids(B, n, K, 1, 9)
    O, _ = _run(Q, Kt, V, ids, window)
    ref = np.zeros_like(O)
    for g in range(K):
        rows = np.nonzero(ids[0, :, 0] == g)[0]
        if len(rows) == 0:
            continue
        r = torch.as_tensor(rows)
        ref[0, rows] = _sdpa(Q[:, r], Kt[:, r], V[:, r], causal=True)[0]
    np.testing.assert_allclose(O, ref, atol=2e-6)


@pytest.mark.parametrize("Hq,Hkv,topk,K,window", [(4, 2, 2, 5, 6), (6, 3, 3, 7, 2), (4, 1, 1, 3, 10)])
def test_explicit_mask_sdpa(Hq, Hkv, topk, K, window):
    """Random ids, GQA: equal to SDPA with the brute-force boolean mask; the
    log-sum-exp equals torch.logsumexp over the masked scores."""
    B, n, d = 2, 100, 64
    Q, Kt, V = _qkv(B, n, Hq, Hkv, d, 41)
    ids = _rand_ids(B, n, K, topk, 13)
    A = _brute_allowed(ids, window)
    O, L = _run(Q, Kt, V, ids, window)
    np.testing.assert_allclose(O, _sdpa(Q, Kt, V, mask=A), atol=2e-6)
    np.testing.assert_allclose(L, _lse(Q, Kt, A), atol=2e-5)


def test_rows_subset_matches_full():
    B, n, H, d = 2, 80, 2, 32
    Q, K, V = _qkv(B, n, H, H, d, 51)
    ids = _rand_ids(B, n, 6, 2, 17)
    O, L = _run(Q, K, V, ids, 5)
    rows = np.array([0, 79, 80, 123, 159, 4], np.int64)
    Os, Ls = _run(Q, K, V, ids, 5, rows=rows)
    np.testing.assert_array_equal(Os, O.reshape(B * n, H, d)[rows])
    np.testing.assert_array_equal(Ls, L.reshape(B * n, H)[rows])


def test_rows_only_q_matches_full_and_sdpa():
    """The sampled-Q form (Q holds only the sampled rows, in the order of
    `rows`): rows from both batches, out of order, agree bit for bit with the
    full-Q call on those rows, and with SDPA under the brute-force mask."""
    B, n, Hq, Hkv, d = 2, 90, 4, 2, 32
    Q, K, V = _qkv(B, n, Hq, Hkv, d, 53)
    ids = _rand_ids(B, n, 5, 2, 29)
    window = 6
    rows = np.array([131, 7, 89, 90, 0, 179, 45, 100], np.int64)
    Qr = Q.reshape(B * n, Hq, d)[torch.as_tensor(rows)]
    Os, Ls = _run(Qr, K, V, ids, window, rows=rows)
    O, L = _run(Q, K, V, ids, window)
    np.testing.assert_array_equal(Os, O.reshape(B * n, Hq, d)[rows])
    np.testing.assert_array_equal(Ls, L.reshape(B * n, Hq)[rows])
    A = _brute_allowed(ids, window)
    ref = _sdpa(Q, K, V, mask=A).reshape(B * n, Hq, d)[rows]
    np.testing.assert_allclose(Os, ref, atol=2e-6)
    lref = _lse(Q, K, A).reshape(B * n, Hq)[rows]
    np.testing.assert_allclose(Ls, lref, atol=2e-5)


def test_rows_sum_to_one():
    B, n, H, d = 1, 64, 2, 16
    Q, K, _ = _qkv(B, n, H, H, d, 61)
    V = torch.ones(B, n, H, d, dtype=torch.bfloat16)
    O, _ = _run(Q, K, V, _rand_ids(B, n, 4, 2, 19), 3)
    np.testing.assert_allclose(O, 1.0, atol=1e-6)


# ------------------------------------------------------------- count pins ---

def test_count_closed_forms():
    n = 200
    i = np.arange(n)
    per, tot = oracle.count_pairs(np.zeros((1, n, 1), np.int32), 7)
    assert (per[0] == i + 1).all() and tot == n * (n + 1) // 2
    per, _ = oracle.count_pairs(np.arange(n, dtype=np.int32).reshape(1, n, 1), 7)
    assert (per[0] == np.minimum(7, i + 1)).all()
    per, _ = oracle.count_pairs(np.arange(n, dtype=np.int32).reshape(1, n, 1), 0)
    assert (per[0] == 1).all()          # only the token itself (its own group)


@pytest.mark.parametrize("window", [0, 3, 11])
def test_count_rows_subset(window):
    """Counting only sampled rows (both batches, out of order) gives the
    brute-force set counts of those rows and their sum."""
    B, n = 2, 70
    ids = _rand_ids(B, n, 6, 2, 31 + window)
    rows = np.array([139, 0, 69, 70, 5, 100, 33], np.int64)
    per, tot = oracle.count_pairs(ids, window, rows=rows)
    A = _brute_allowed(ids, window).reshape(B * n, n)
    expect = A[rows].sum(-1)
    np.testing.assert_array_equal(per, expect)
    assert tot == int(expect.sum())
    full, _ = oracle.count_pairs(ids, window)
    np.testing.assert_array_equal(per, full.reshape(-1)[rows])


# ------------------------------------------------------------ assign pins ---

def test_assign_closed_form_identity_projection():
    """hidden = d_g, W_g = I, C = I: the scores are x itself, so the top-k is
    the k largest entries of x, ties to the lower index."""
    x = np.array([[0.5, 2.0, -1.0, 2.0, 3.0], [1.0, 1.0, 1.0, 1.0, 1.0],
                  [-4.0, -3.0, -2.0, -1.0, -0.5]], np.float32)
    ids, margin, scores = oracle.assign(_bf16_bits(x), np.eye(5, dtype=np.float32),
                                        np.eye(5, dtype=np.float32), 2)
    assert ids.tolist() == [[4, 1], [0, 1], [4, 3]]
    np.testing.assert_array_equal(scores, x)
    np.testing.assert_allclose(margin, [0.0, 0.0, 0.5])


def test_assign_duplicate_centroid_tie_goes_to_lower_id():
    rng = np.random.default_rng(3)
    C = rng.standard_normal((6, 8)).astype(np.float32)
    C[4] = C[1]
    X = _bf16_bits(rng.standard_normal((50, 8)))
    ids, margin, scores = oracle.assign(X, np.eye(8, dtype=np.float32), C, 6)
    for t in range(50):
        order = list(ids[t])
        assert order.index(1) < order.index(4)


def test_assign_matches_numpy_argsort():
    rng = np.random.default_rng(5)
    hidden, dg, K, topk = 96, 24, 20, 3
    X = _rand_bf16((2, 30, hidden), 77)
    Wg = (rng.standard_normal((hidden, dg)) / np.sqrt(hidden)).astype(np.float32)
    C = rng.standard_normal((K, dg)).astype(np.float32)
    ids, margin, scores = oracle.assign(synth.bits(X), Wg, C, topk)
    s = (X.double().numpy() @ Wg.astype(np.float64)) @ C.astype(np.float64).T
    np.testing.assert_allclose(scores, s, rtol=1e-6, atol=1e-6)
    order = np.argsort(-scores, axis=-1, kind="stable")[..., :topk]
    np.testing.assert_array_equal(ids, order)
    srt = -np.sort(-scores, axis=-1)[..., :topk + 1]
    np.testing.assert_allclose(margin, np.min(srt[..., :-1] - srt[..., 1:], axis=-1))


def test_assign_ranking_invariant_to_positive_scale():
    rng = np.random.default_rng(8)
    X = _rand_bf16((40, 32), 99)
    Wg = rng.standard_normal((32, 16)).astype(np.float32)
    C = rng.standard_normal((10, 16)).astype(np.float32)
    a, _, _ = oracle.assign(synth.bits(X), Wg, C, 4)
    b, _, _ = oracle.assign(synth.bits(X), Wg * 2, C * 0.5, 4)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------ bucket pins ---

@pytest.mark.parametrize("B,n,K,topk", [(2, 257, 7, 2), (1, 33, 40, 1), (3, 100, 4, 4)])
def test_bucket_matches_numpy(B, n, K, topk):
    ids = _rand_ids(B, n, K, topk, 23)
    off, pos, inv = oracle.bucket(ids, K)
    for b in range(B):
        cnt = np.bincount(ids[b].ravel(), minlength=K)
        np.testing.assert_array_equal(off[b], np.concatenate([[0], np.cumsum(cnt)]))
        for g in range(K):
            members = np.nonzero((ids[b] == g).any(-1))[0]
            np.testing.assert_array_equal(pos[b, off[b, g]:off[b, g + 1]], members)
        flat_tok = np.repeat(np.arange(n), topk)
        np.testing.assert_array_equal(pos[b][inv[b].ravel()], flat_tok)
        grp = np.searchsorted(off[b], inv[b].ravel(), side="right") - 1
        np.testing.assert_array_equal(grp, ids[b].ravel())


# ---------------------------------------------------------------- Sinkhorn

def _rand_affinities(B, n, K, seed, scale=2.0):
    r = np.random.default_rng(seed)
    return (scale * r.standard_normal((B, n, K))).astype(np.float32)


def test_sinkhorn_hand_worked_example():
    """One round on a 2 x 2 matrix, worked by hand (tests/golden)."""
    g = json.load(open(os.path.join(GOLDEN, "sinkhorn_2x2.json")))
    S = np.array([[[0.0, np.log(2.0)], [np.log(3.0), 0.0]]], np.float32)
    P, lu, lv = oracle.sinkhorn(S, g["tau"], g["iters"])
    # S holds ln 2 and ln 3 rounded to float32: agreement to ~1e-7
    np.testing.assert_allclose(P[0], np.array(g["P"]), atol=2e-7)
    np.testing.assert_allclose(lu[0], np.array(g["log_u"]), atol=2e-7)
    np.testing.assert_allclose(lv[0], np.array(g["log_v"]), atol=2e-7)


@pytest.mark.parametrize("iters", [1, 2, 7])
def test_sinkhorn_rank_one_closed_form(iters):
    """S_ic = alpha_i + beta_c (a rank-one kernel) is balanced by one round:
    P = 1/K everywhere, whatever alpha and beta."""
    r = np.random.default_rng(5)
    n, K = 37, 6
    S = (r.standard_normal((n, 1)) * 3 + r.standard_normal((1, K)) * 3).astype(np.float32)
    P, _, _ = oracle.sinkhorn(S[None], 1.0, iters)
    np.testing.assert_allclose(P[0], 1.0 / K, rtol=1e-5)


@pytest.mark.parametrize("n,K", [(50, 4), (7, 13), (300, 64)])
def test_sinkhorn_marginals(n, K):
    """After every round the group masses are exactly n / K (the last
    update); with many rounds the token masses converge to 1."""
    S = _rand_affinities(2, n, K, seed=n + K)
    P, _, _ = oracle.sinkhorn(S, 1.0, 1)
    np.testing.assert_allclose(P.sum(axis=1), n / K, rtol=1e-12)
    P, _, _ = oracle.sinkhorn(S, 1.0, 400)
    np.testing.assert_allclose(P.sum(axis=1), n / K, rtol=1e-12)
    np.testing.assert_allclose(P.sum(axis=2), 1.0, atol=1e-9)


def test_sinkhorn_row_shift_and_temperature():
    """A constant added to a token's row is absorbed by its u (P unchanged at
    any round count); S / tau at tau = 1 equals S at temperature tau."""
    S = _rand_affinities(1, 40, 8, seed=3)
    shift = np.random.default_rng(4).standard_normal((1, 40, 1)).astype(np.float32) * 5
    P0, _, _ = oracle.sinkhorn(S, 1.0, 3)
    P1, _, _ = oracle.sinkhorn((S + shift).astype(np.float32), 1.0, 3)
    np.testing.assert_allclose(P1, P0, rtol=1e-5, atol=1e-9)
    Pt, _, _ = oracle.sinkhorn(S, 0.5, 3)
    Ps, _, _ = oracle.sinkhorn((S / 0.5).astype(np.float32), 1.0, 3)
    np.testing.assert_allclose(Pt, Ps, rtol=1e-12)


def test_sinkhorn_permutations_and_batch():
    """Permuting tokens or groups permutes P alike; each sequence of a batch
    is normalised on its own."""
    S = _rand_affinities(2, 30, 5, seed=8)
    P, lu, lv = oracle.sinkhorn(S, 1.0, 4)
    pt = np.random.default_rng(1).permutation(30)
    pg = np.random.default_rng(2).permutation(5)
    Pp, _, _ = oracle.sinkhorn(np.ascontiguousarray(S[:, pt][:, :, pg]), 1.0, 4)
    np.testing.assert_allclose(Pp, P[:, pt][:, :, pg], rtol=1e-12)
    P1, lu1, lv1 = oracle.sinkhorn(S[1:], 1.0, 4)
    np.testing.assert_allclose(P1[0], P[1], rtol=1e-12)
    np.testing.assert_allclose(lu1[0], lu[1], rtol=1e-12)
    np.testing.assert_allclose(lv1[0], lv[1], rtol=1e-12)


def test_sinkhorn_matches_multiplicative_scaling():
    """The log-domain rounds against the plain multiplicative form of the
    same scaling (u = a / (A v), v = b / (A^T u)) on a well-scaled problem."""
    S = _rand_affinities(1, 20, 6, seed=11, scale=1.0)
    P, _, _ = oracle.sinkhorn(S, 1.0, 5)
    A = np.exp(S[0].astype(np.float64))
    v = np.ones(6)
    for _ in range(5):
        u = 1.0 / (A @ v)
        v = (20 / 6) / (A.T @ u)
    np.testing.assert_allclose(P[0], u[:, None] * A * v[None, :], rtol=1e-10)


# ------------------------------------------------- soft-gated attention (training)

def _grid_bf16(shape, seed, step=2.0 ** -7, span=200):
    """Values m * step with |m| < span: exact in bf16, and so are x +- step."""
    r = np.random.default_rng(seed)
    return (r.integers(-span, span, size=shape) * step).astype(np.float32)


def _bits_of(x):
    return synth.bits(torch.from_numpy(x).to(torch.bfloat16))


def _sdpa64(Q, K, V, scale):
    """Causal SDPA in float64 with torch, [B, n, H, d] layout, GQA expanded."""
    q = torch.from_numpy(Q).double().transpose(1, 2)
    grp = Q.shape[2] // K.shape[2]
    k = torch.from_numpy(K).double().repeat_interleave(grp, dim=2).transpose(1, 2)
    v = torch.from_numpy(V).double().repeat_interleave(grp, dim=2).transpose(1, 2)
    return q, k, v


@pytest.mark.parametrize("window,lam,scale_mul", [
    (10 ** 6, 3.0, 1.0),    # every pair local: gate 1, plain causal attention
    (0, 0.0, 0.5),          # no pair local, lambda 0: gate 1/2 everywhere
])
def test_gated_reduces_to_causal_sdpa(window, lam, scale_mul):
    B, n, Hq, Hkv, d, Kg = 2, 23, 4, 2, 16, 5
    Q = _grid_bf16((B, n, Hq, d), 1)
    K = _grid_bf16((B, n, Hkv, d), 2)
    V = _grid_bf16((B, n, Hkv, d), 3)
    G = np.random.default_rng(4).random((B, n, Kg)).astype(np.float32)
    dO = np.random.default_rng(5).standard_normal((B, n, Hq, d)).astype(np.float32)
    O, L = oracle.gated_fwd(_bits_of(Q), _bits_of(K), _bits_of(V), G, window, lam)
    dQ, dK, dV, dG, dl = oracle.gated_bwd(_bits_of(Q), _bits_of(K), _bits_of(V), G, dO, window,
                                          lam)
    q, k, v = _sdpa64(Q, K, V, 1.0)
    q.requires_grad_(True)
    k.requires_grad_(True)
    v.requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                         scale=scale_mul / np.sqrt(d))
    np.testing.assert_allclose(O, o.detach().transpose(1, 2).numpy(), atol=1e-12)
    (o * torch.from_numpy(dO).double().transpose(1, 2)).sum().backward()
    grp = Hq // Hkv
    np.testing.assert_allclose(dQ, q.grad.transpose(1, 2).numpy(), atol=1e-11)
    dk = k.grad.transpose(1, 2).numpy().reshape(B, n, Hkv, grp, d).sum(3)
    dv = v.grad.transpose(1, 2).numpy().reshape(B, n, Hkv, grp, d).sum(3)
    np.testing.assert_allclose(dK, dk, atol=1e-11)
    np.testing.assert_allclose(dV, dv, atol=1e-11)
    if window >= n:   # no gate anywhere: nothing flows to G or lambda
        assert np.abs(dG).max() == 0.0 and dl == 0.0


def test_gated_saturated_gate_is_plain_attention():
    """lambda large with every affinity >= 0.5: sigma(lambda a) rounds to 1 in
    double, so the result is causal attention whatever the window."""
    B, n, Hq, Hkv, d, Kg = 1, 17, 2, 2, 8, 4
    Q, K, V = _grid_bf16((B, n, Hq, d), 6), _grid_bf16((B, n, Hkv, d), 7), _grid_bf16((B, n, Hkv, d), 8)
    G = np.full((B, n, Kg), 0.5, np.float32)   # a_ij = 1
    O, _ = oracle.gated_fwd(_bits_of(Q), _bits_of(K), _bits_of(V), G, 3, 80.0)
    q, k, v = _sdpa64(Q, K, V, 1.0)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                         scale=1 / np.sqrt(d))
    np.testing.assert_allclose(O, o.transpose(1, 2).numpy(), atol=1e-12)


def test_gated_gradients_by_finite_differences():
    """Central differences of L = sum(O * dO) with steps exact in bf16 (Q, K,
    V on a 2^-7 grid), in float32 (G) and in double (lambda), against every
    gradient of the backward, on a case with local and gated pairs."""
    B, n, Hq, Hkv, d, Kg, window, lam = 1, 9, 2, 1, 4, 3, 3, 2.5
    h = 2.0 ** -7
    Q, K, V = _grid_bf16((B, n, Hq, d), 11), _grid_bf16((B, n, Hkv, d), 12), _grid_bf16((B, n, Hkv, d), 13)
    G = (np.random.default_rng(14).integers(1, 100, size=(B, n, Kg)) * 2.0 ** -7).astype(np.float32)
    dO = np.random.default_rng(15).standard_normal((B, n, Hq, d)).astype(np.float32)

    def loss(Qx=Q, Kx=K, Vx=V, Gx=G, lx=lam):
        O, _ = oracle.gated_fwd(_bits_of(Qx), _bits_of(Kx), _bits_of(Vx), Gx, window, lx)
        return float((O * dO).sum())

    dQ, dK, dV, dG, dl = oracle.gated_bwd(_bits_of(Q), _bits_of(K), _bits_of(V), G, dO, window,
                                          lam)
    for name, X, grad in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV), ("G", G, dG)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = dict(Qx=Q, Kx=K, Vx=V, Gx=G)
            args_m = dict(Qx=Q, Kx=K, Vx=V, Gx=G)
            args_p[name + "x"], args_m[name + "x"] = Xp, Xm
            num[idx] = (loss(**args_p) - loss(**args_m)) / (2 * h)
        err = np.abs(num - grad).max()
        assert err <= 2e-3 * max(1.0, np.abs(grad).max()), (name, err)
    numl = (loss(lx=lam + 1e-5) - loss(lx=lam - 1e-5)) / 2e-5
    assert abs(numl - dl) <= 1e-6 * max(1.0, abs(dl)), (numl, dl)
