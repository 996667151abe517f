"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side validation rejects bad arguments before any CUDA call
(no GPU needed: the fake pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "focus.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
P = ctypes.c_void_p(0x10000)        # aligned, never dereferenced
P2 = ctypes.c_void_p(0x20000)
MIS = ctypes.c_void_p(0x10004)      # misaligned


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fg.library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(focus_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_path_calls():
    names = _declared()
    for n in ("focus_assign", "focus_bucket", "focus_attention_fwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert fg.focus_status_string(0) == "FOCUS_OK"
    assert fg.focus_status_string(3) == "FOCUS_ERR_WORKSPACE"
    assert "sm_103a" in fg.focus_version()


def test_assign_validation(lib):
    f = lib.focus_assign
    need = fg.focus_assign_workspace_size(1, 8, 64, 16, 8, 2)
    assert need > 0
    assert fg.focus_assign_workspace_size(1, 8, 64, 16, 300, 2) == 0   # K > 256: fp32 kernel
    # more centroids than centroid dimensions: Z = X W_g is kept per token
    z1 = fg.focus_assign_workspace_size(1, 1000, 64, 64, 256, 2)
    z2 = fg.focus_assign_workspace_size(2, 1000, 64, 64, 256, 2)
    assert z2 - z1 >= 1000 * (2 * 64 * 2 + 4)      # fp16 hi + lo of 64 values, a scale

    def call(X=P, hid=64, dg=16, K=8, topk=2, ws=P2, nbytes=need):
        #        X  Wg C  B  n  hidden dg  K  topk ids margin ws  bytes  stream
        return f(X, P, P, 1, 8, hid, dg, K, topk, P, None, ws, nbytes, None)

    assert call(X=None) == INVALID
    assert call(topk=9) == INVALID                      # topk > K
    assert call(topk=0) == INVALID
    assert call(X=MIS) == INVALID
    assert call(hid=60) == UNSUPPORTED                  # hidden % 8
    assert call(dg=300) == UNSUPPORTED                  # d_g > 256
    assert call(K=2000) == UNSUPPORTED                  # K > 1024
    assert call(K=20, topk=9) == UNSUPPORTED            # topk > 8
    assert call(nbytes=need - 1) == WORKSPACE
    assert call(ws=None) == WORKSPACE


def test_bucket_validation(lib):
    f = lib.focus_bucket
    need = fg.focus_bucket_workspace_size(2, 5000, 64, 2)
    assert need > 0
    assert f(None, 2, 5000, 64, 2, P, P, P, P, need, None) == INVALID
    assert f(P, 2, 5000, 64, 65, P, P, P, P, need, None) == INVALID          # topk > K
    assert f(P, 2, 5000, 64, 2, P, P, P, P, need - 1, None) == WORKSPACE
    assert f(P, 2, 5000, 64, 2, P, P, P, None, need, None) == INVALID
    assert f(P, 2, 5000, 2048, 2, P, P, P, P, 1 << 40, None) == UNSUPPORTED


def test_attention_validation(lib):
    f = lib.focus_attention_fwd
    need = fg.focus_attention_workspace_size(1, 1000, 8, 2, 128, 16, 2)
    assert need > 0

    def call(Q=P, Hq=8, Hkv=2, d=128, window=16, K=16, topk=2, ws=P, nbytes=need, n=1000, B=1):
        return f(Q, P, P, B, n, Hq, Hkv, d, window, 0.0, P, P, P, P, K, topk, P2, None, ws,
                 nbytes, None)

    assert call(Q=None) == INVALID
    assert call(Q=MIS) == INVALID
    assert call(Hq=8, Hkv=3) == INVALID                  # Hq % Hkv
    assert call(window=-1) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(topk=17) == INVALID                      # topk > K
    assert call(K=2000, topk=2) == UNSUPPORTED
    # every documented shape fits the kernels' shared memory, up to K = 1024
    # and topk = 8 at d = 128 (supported shapes then stop at the workspace
    # check: nothing launches)
    assert call(d=128, K=1024, topk=1, nbytes=1) == WORKSPACE
    assert call(d=128, K=1024, topk=8, nbytes=1) == WORKSPACE
    assert call(d=64, K=1024, topk=8, nbytes=1) == WORKSPACE
    assert call(d=128, K=1025, topk=8, nbytes=1) == UNSUPPORTED
    assert call(nbytes=need - 1) == WORKSPACE
    assert call(ws=None) == INVALID
    assert call(n=0) == INVALID


def test_attention_workspace_grows_with_problem(lib):
    a = fg.focus_attention_workspace_size(1, 1024, 8, 8, 64, 16, 1)
    b = fg.focus_attention_workspace_size(1, 2048, 8, 8, 64, 16, 1)
    c = fg.focus_attention_workspace_size(1, 2048, 8, 8, 64, 16, 2)
    assert 0 < a < b < c
    assert fg.focus_attention_workspace_size(0, 2048, 8, 8, 64, 16, 2) == 0


def test_dense_and_count_validation(lib):
    assert lib.focus_dense_causal_fwd(None, P, P, 1, 64, 2, 2, 64, 0.0, P2, None, None) == INVALID
    assert lib.focus_dense_causal_fwd(P, P, P, 1, 64, 2, 2, 80, 0.0, P2, None, None) == UNSUPPORTED
    assert lib.focus_dense_causal_fwd(P, P, P, 1, 64, 3, 2, 64, 0.0, P2, None, None) == INVALID
    assert lib.focus_count_pairs(P, P, P, P, 1, 64, 8, 2, 4, None, None, None) == INVALID
    assert lib.focus_count_pairs(P, P, P, P, 1, 64, 8, 2, -1, None, P, None) == INVALID


def test_sinkhorn_validation(lib):
    f = lib.focus_sinkhorn
    need = fg.focus_sinkhorn_workspace_size(2, 1000, 64)
    assert need >= 2 * 64 * 4 + 2 * 1000 * 4
    assert fg.focus_sinkhorn_workspace_size(1, 10, 1025) == 0       # K above 1024
    assert fg.focus_sinkhorn_workspace_size(1, 0, 8) == 0
    ok = (P, 2, 1000, 64, 1.0, 3, P2, P2, P2, P2, need, None)
    for k, bad in ((0, None), (0, MIS), (1, 0), (2, 0), (3, 0), (3, 1025), (4, -1.0),
                   (4, float("nan")), (5, 0), (6, MIS), (7, MIS), (8, MIS), (9, None),
                   (9, MIS)):
        args = list(ok)
        args[k] = bad
        assert f(*args) == INVALID, (k, bad)
    args = list(ok)
    args[10] = need - 1
    assert f(*args) == WORKSPACE


def test_gated_validation(lib):
    need = fg.focus_gated_workspace_size(1, 100, 4, 2, 16)
    assert need > 0
    assert fg.focus_gated_workspace_size(1, 100, 4, 2, 129) == 0   # K_g above 128
    assert fg.focus_gated_workspace_size(1, 100, 4, 3, 16) == 0    # Hq % Hkv != 0
    f = lib.focus_gated_attention_fwd
    ok = (P, P, P, P, 1, 100, 4, 2, 64, 16, 8, 2.0, 0.0, P2, P2, P2, need, None)
    for k, bad, want in ((0, None, INVALID), (3, MIS, INVALID), (4, 0, INVALID),
                         (7, 3, INVALID), (8, 96, UNSUPPORTED), (9, 129, UNSUPPORTED),
                         (10, -1, INVALID), (11, float("inf"), INVALID), (12, -1.0, INVALID),
                         (13, None, INVALID), (14, MIS, INVALID), (16, need - 1, WORKSPACE)):
        args = list(ok)
        args[k] = bad
        assert f(*args) == want, (k, bad)
    g = lib.focus_gated_attention_bwd
    okb = (P, P, P, P, P, P, P, 1, 100, 4, 2, 64, 16, 8, 2.0, 0.0, P2, P2, P2, P2, P2, P2, need,
           None)
    for k, bad, want in ((4, None, INVALID), (6, MIS, INVALID), (16, None, INVALID),
                         (20, None, INVALID), (12, 0, INVALID), (22, need - 1, WORKSPACE)):
        args = list(okb)
        args[k] = bad
        assert g(*args) == want, (k, bad)


def test_prefill_validation(lib):
    f = lib.focus_prefill
    need = fg.focus_prefill_workspace_size(1, 512, 64, 4, 4, 64, 16, 8, 2, 0)
    need_host = fg.focus_prefill_workspace_size(1, 512, 64, 4, 4, 64, 16, 8, 2, 1)
    assert need_host > need > 0
    args = [P, P, P, P, P, P, 1, 512, 64, 4, 4, 64, 16, 8, 2, 16, 0.0, P2, None, None, P]
    assert f(*args, need - 1, 0, None) == WORKSPACE
    bad = list(args)
    bad[11] = 72      # d
    assert f(*bad, need, 0, None) == UNSUPPORTED
    bad = list(args)
    bad[0] = None
    assert f(*bad, need, 0, None) == INVALID


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle (test infrastructure only)."""
    pkg = os.path.join(ROOT, "learned_group_sparse_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
