"""Decode parity: one new token per sequence against a key/value cache whose
group memberships are kept as per-group position lists.  Each step's output
is compared with the oracle's masked-softmax attention for that token (the
last row of the cache), and the lists grown by the appends are compared bit
for bit with the oracle's bucketing of the whole cache."""
import numpy as np
import pytest
import torch

import oracle
import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build, synth
from _gpu_helpers import check_output, free_cuda

pytestmark = pytest.mark.gpu

CAPACITY = 6   # FOCUS_ERR_CAPACITY


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    fg.focus_get_device_status(reset=True)
    yield
    assert fg.focus_get_device_status(reset=True) == 0, "device status set"
    free_cuda()


def _rand_ids(B, n, K, topk, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    r = torch.rand(B * n, K, generator=g, device="cuda")
    return torch.topk(r, topk, dim=1).indices.to(torch.int32).view(B, n, topk).contiguous()


def _cache(B, L, Hq, Hkv, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    Q = torch.randn(B, L, Hq, d, generator=g, device="cuda", dtype=torch.bfloat16)
    K = torch.randn(B, L, Hkv, d, generator=g, device="cuda", dtype=torch.bfloat16)
    V = torch.randn(B, L, Hkv, d, generator=g, device="cuda", dtype=torch.bfloat16)
    return Q, K, V


def _check_lists(glen, gpos, ids_np, K):
    off, pos, _ = oracle.bucket(ids_np, K)
    gl, gp = glen.cpu().numpy(), gpos.cpu().numpy()
    B = ids_np.shape[0]
    for b in range(B):
        sizes = np.diff(off[b])
        np.testing.assert_array_equal(gl[b], sizes)
        for g in range(K):
            np.testing.assert_array_equal(gp[b, g, :sizes[g]], pos[b, off[b, g]:off[b, g + 1]])


DECODE_CASES = [
    # B, prefix n, steps, Hq, Hkv, d, K, topk, window
    (2, 700, 6, 4, 1, 128, 16, 2, 64),
    (1, 300, 5, 2, 2, 64, 5, 3, 0),       # no window: group keys only (the token itself too)
    (2, 513, 4, 8, 1, 128, 8, 8, 16),     # topk = K: every pair shares group 0
    (1, 400, 4, 6, 3, 64, 32, 1, 1000),   # the window covers the whole cache
    (3, 257, 3, 32, 8, 128, 64, 2, 128),  # GQA 4:1
    (1, 0, 5, 4, 2, 128, 4, 2, 2),        # no prefix: every list starts empty
    (152, 3000, 2, 2, 1, 64, 4, 2, 256),  # 152 sequences: one split each, several mapping passes
    (40, 3000, 2, 8, 8, 64, 4, 2, 256),   # four splits of 8 kv heads each
    (19, 3000, 2, 16, 8, 128, 8, 3, 64),  # eight splits, d = 128
]


@pytest.mark.parametrize("case", DECODE_CASES,
                         ids=lambda c: "B{}n{}s{}H{}x{}d{}K{}k{}w{}".format(*c))
def test_decode_steps_match_oracle(case):
    B, n, steps, Hq, Hkv, d, K, topk, window = case
    Lmax = n + steps
    ids = _rand_ids(B, Lmax, K, topk, seed=n + K)
    Qall, Kc, Vc = _cache(B, Lmax, Hq, Hkv, d, seed=3 * n + d)
    ids_np = ids.cpu().numpy()
    if n:
        off, pos, _ = fg.focus_bucket(ids[:, :n].contiguous(), K)
    else:   # an empty prefix: every group empty
        off = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
        pos = torch.empty(B, 0, dtype=torch.int32, device="cuda")
    glen, gpos = fg.focus_decode_lists_init(off, pos, K, topk, cap=Lmax)
    for L in range(n + 1, Lmax + 1):
        q = Qall[:, L - 1].contiguous()
        O, lse = fg.focus_decode_fwd(q, Kc, Vc, ids, L, window, glen, gpos, K)
        torch.cuda.synchronize()
        rows = np.array([b * L + L - 1 for b in range(B)], np.int64)
        Oref, Lref = oracle.attention(synth.bits(q), synth.bits(Kc[:, :L].contiguous()),
                                      synth.bits(Vc[:, :L].contiguous()), ids_np[:, :L],
                                      window, rows=rows)
        check_output(O, Oref, lse, Lref, label=f"{case} L={L}")
    _check_lists(glen, gpos, ids_np, K)


def test_decode_at_one_million_tokens():
    """The n = 1M workload's shapes (GQA 32/8, d 128, K 256, top-2, window
    1024) with seeded ids of the assignment's structure: one decode step for
    the last token, over lists built from the first n - 1 tokens."""
    w = synth.workload(4)
    n = w.n
    comp = synth.make_components(w, "cuda")
    ids = synth.synthetic_ids(w, comp, "cuda")
    _, Kc, Vc = synth.make_qkv(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(77)
    q = torch.randn(w.B, w.Hq, w.d, generator=g, device="cuda", dtype=torch.bfloat16)
    off, pos, _ = fg.focus_bucket(ids[:, :n - 1].contiguous(), w.K)
    cap = int((off[:, 1:] - off[:, :-1]).max()) + 16
    glen, gpos = fg.focus_decode_lists_init(off, pos, w.K, w.topk, cap=cap)
    O, lse = fg.focus_decode_fwd(q, Kc, Vc, ids, n, w.window, glen, gpos, w.K)
    torch.cuda.synchronize()
    ids_np = ids.cpu().numpy()
    Oref, Lref = oracle.attention(synth.bits(q), synth.bits(Kc), synth.bits(Vc), ids_np,
                                  w.window, rows=np.array([n - 1], np.int64))
    check_output(O, Oref, lse, Lref, label="decode n1m")
    # the new token now heads the end of its groups' lists
    gl = glen.cpu().numpy()[0]
    for gid in ids_np[0, n - 1]:
        assert int(gpos[0, gid, gl[gid] - 1]) == n - 1
    del Kc, Vc
    free_cuda()


def test_list_capacity_overflow_is_reported():
    """A list already holding cap members is not appended to, and the
    device status word reads FOCUS_ERR_CAPACITY."""
    B, n, K, topk = 1, 40, 2, 1
    ids = torch.zeros(B, n + 1, topk, dtype=torch.int32, device="cuda")   # one group
    off, pos, _ = fg.focus_bucket(ids[:, :n].contiguous(), K)
    glen, gpos = fg.focus_decode_lists_init(off, pos, K, topk, cap=n)
    assert fg.focus_get_device_status(reset=True) == 0
    q, Kc, Vc = _cache(B, n + 1, 2, 2, 64, seed=9)
    fg.focus_decode_fwd(q[:, n].contiguous(), Kc, Vc, ids, n + 1, 4, glen, gpos, K)
    assert fg.focus_get_device_status(reset=True) == CAPACITY
    assert int(glen[0, 0]) == n
