"""GPU parity at the five workload sizes, in the launch configuration the
benchmark times (focus_assign, focus_bucket, focus_attention_fwd with
full-size buffers).  Small workloads are compared on every output; large
ones on seeded sampled rows that always include the first and last rows,
the window edge and members of the largest and smallest groups."""
import numpy as np
import pytest
import torch

import oracle
import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build, synth
from _gpu_helpers import check_ids, check_output, free_cuda, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    fg.focus_get_device_status(reset=True)
    yield
    assert fg.focus_get_device_status(reset=True) == 0, "a device-side wait timed out"
    free_cuda()


FULL_ORACLE_TOKENS = 8192   # up to this many tokens every output row is checked


@pytest.mark.parametrize("idx", range(len(synth.WORKLOADS)), ids=[w.name for w in synth.WORKLOADS])
def test_workload(idx):
    w = synth.workload(idx)
    ntok = w.B * w.n
    rng = np.random.default_rng(idx)
    Wg, C = synth.make_params(w, "cuda")
    comp = synth.make_components(w, "cuda")

    # ---- assignment: every token (small) or 4096 sampled tokens (large)
    X = synth.make_x(w, Wg, C, comp, "cuda")
    ids_gpu, _ = fg.focus_assign(X, Wg, C, w.topk)
    torch.cuda.synchronize()
    tok = np.arange(ntok) if ntok <= FULL_ORACLE_TOKENS else \
        np.sort(rng.choice(ntok, size=4096, replace=False))
    Xh = synth.bits(X.view(ntok, w.hidden)[torch.from_numpy(tok).cuda()])
    rids, rmargin, _ = oracle.assign(Xh, Wg.cpu().numpy(), C.cpu().numpy(), w.topk)
    skipped = check_ids(ids_gpu.view(ntok, w.topk)[torch.from_numpy(tok).cuda()], rids, rmargin)
    assert skipped <= max(4, len(tok) // 50), skipped
    del X, ids_gpu
    free_cuda()

    # ---- attention on ids both sides share: the oracle's own ids for the
    # small workloads, seeded synthetic ids (same structure) for the large
    if ntok <= FULL_ORACLE_TOKENS:
        ids_np = rids.reshape(w.B, w.n, w.topk)
    else:
        ids_np = synth.synthetic_ids(w, comp, "cuda").cpu().numpy()
    Q, K, V = synth.make_qkv(w, "cuda")
    ids = torch.from_numpy(ids_np).cuda()
    off, pos, inv = fg.focus_bucket(ids, w.K)
    O, L = fg.focus_attention_fwd(Q, K, V, w.window, ids, off, pos, inv, w.K)
    torch.cuda.synchronize()
    if ntok <= FULL_ORACLE_TOKENS:
        Oref, Lref = oracle.attention(synth.bits(Q), synth.bits(K), synth.bits(V), ids_np,
                                      w.window)
        check_output(O, Oref, L.permute(0, 2, 1), Lref, label=w.name)
    else:
        rows = sample_rows(w.B, w.n, w.window, ids_np, seed=idx)
        rt = torch.from_numpy(rows).cuda()
        Qr = synth.bits(Q.view(ntok, w.Hq, w.d)[rt])
        Oref, Lref = oracle.attention(Qr, synth.bits(K), synth.bits(V), ids_np, w.window,
                                      rows=rows)
        Og = O.view(ntok, w.Hq, w.d)[rt]
        Lg = L.permute(0, 2, 1).reshape(ntok, w.Hq)[rt]
        check_output(Og, Oref, Lg, Lref, label=w.name)

    # ---- every allowed pair scored exactly once
    _, _, cnt = fg.focus_attention_fwd_counted(Q, K, V, w.window, ids, off, pos, inv, w.K)
    per, tot = fg.focus_count_pairs(ids, off, pos, inv, w.K, w.window)
    torch.cuda.synchronize()
    assert torch.equal(cnt.long(), per)
    if ntok <= 4 * FULL_ORACLE_TOKENS * 2:
        rper, rtot = oracle.count_pairs(ids_np, w.window)
        np.testing.assert_array_equal(per.cpu().numpy(), rper)
        assert int(tot[0]) == rtot
    else:
        # the sampled rows: both the count kernel and the counted attention
        # against the oracle's enumeration of the rule
        rper, _ = oracle.count_pairs(ids_np, w.window, rows=rows)
        np.testing.assert_array_equal(per.view(-1)[rt].cpu().numpy(), rper)
        np.testing.assert_array_equal(cnt.view(-1)[rt].long().cpu().numpy(), rper)
    del Q, K, V, O, L
    free_cuda()
