"""The bounded device-side waits' error path, exercised without faulting or
hanging the GPU: with the wait limit set to a nanosecond, the waits of the
next launches run out, the kernels finish early (letting the copies and
tensor-core operations they issued land), and the device status word reads
FOCUS_ERR_TIMEOUT.  Afterwards, with the default limit back, the same call
gives its normal, bit-identical result."""
import pytest
import torch

import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build, synth

pytestmark = pytest.mark.gpu

TIMEOUT = 5   # FOCUS_ERR_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    fg.focus_get_device_status(reset=True)
    yield
    fg.focus_set_wait_limit(0)
    assert fg.focus_get_device_status(reset=True) == 0
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", [
    # tensor-core assignment in the order X (W_g C^T), attention, merge
    synth.small(B=1, n=4096, hidden=1024, Hq=4, Hkv=2, d=128, K=16, dg=64, topk=2, window=256,
                seed=31),
    # assignment in the order (X W_g) C^T (GEMM and scoring kernels)
    synth.small(B=1, n=3000, hidden=512, Hq=2, Hkv=2, d=64, K=200, dg=64, topk=2, window=64,
                seed=32),
], ids=["xm", "xw_c"])
def test_wait_timeout_reported_then_recovered(w):
    t = synth.make_all(w, "cuda")
    ids = torch.empty(w.B, w.n, w.topk, dtype=torch.int32, device="cuda")

    def run():
        O, _ = fg.focus_prefill(t["X"], t["Wg"], t["C"], t["Q"], t["K"], t["V"], w.topk,
                                w.window, ids_out=ids)
        return O

    O_ref = run()
    ids_ref = ids.clone()
    assert fg.focus_get_device_status(reset=True) == 0
    fg.focus_set_wait_limit(1)
    try:
        run()
        st = fg.focus_get_device_status(reset=True)
    finally:
        fg.focus_set_wait_limit(0)
    assert st == TIMEOUT
    O = run()
    assert fg.focus_get_device_status(reset=True) == 0
    assert torch.equal(ids, ids_ref)
    assert torch.equal(O, O_ref)


def test_decode_wait_timeout_reported_then_recovered():
    """The decode attention's copy ring (bulk copies into shared memory, waits
    on full and empty barriers) gives up on the one-nanosecond limit, lets its
    copies land and reports FOCUS_ERR_TIMEOUT; with the limit back the same
    step (lists restored) gives its normal result.  Four groups over 200K
    tokens give every CTA about eighty stages, so that some wait has to wait."""
    B, n, Hq, Hkv, d, K, topk, window = 1, 200000, 8, 8, 128, 4, 2, 128
    g = torch.Generator(device="cuda").manual_seed(41)
    ids = torch.topk(torch.rand(B * n, K, generator=g, device="cuda"), topk, dim=1).indices
    ids = ids.to(torch.int32).view(B, n, topk).contiguous()
    Kc = torch.randn(B, n, Hkv, d, generator=g, device="cuda", dtype=torch.bfloat16)
    Vc = torch.randn(B, n, Hkv, d, generator=g, device="cuda", dtype=torch.bfloat16)
    q = torch.randn(B, Hq, d, generator=g, device="cuda", dtype=torch.bfloat16)
    off, pos, _ = fg.focus_bucket(ids[:, :n - 1].contiguous(), K)
    glen, gpos = fg.focus_decode_lists_init(off, pos, K, topk, cap=n)
    glen0 = glen.clone()

    def run():
        glen.copy_(glen0)
        O, _ = fg.focus_decode_fwd(q, Kc, Vc, ids, n, window, glen, gpos, K)
        return O

    O_ref = run()
    torch.cuda.synchronize()
    assert fg.focus_get_device_status(reset=True) == 0
    fg.focus_set_wait_limit(1)
    try:
        run()
        st = fg.focus_get_device_status(reset=True)
    finally:
        fg.focus_set_wait_limit(0)
    assert st == TIMEOUT
    O = run()
    assert fg.focus_get_device_status(reset=True) == 0
    assert torch.equal(O, O_ref)


def test_sinkhorn_wait_timeout_reported_then_recovered():
    """The Sinkhorn sweep's bulk-copy ring gives up on the one-nanosecond
    limit (the whole CTA leaves at its next barrier after letting the copies
    land) and reports FOCUS_ERR_TIMEOUT; with the limit back the same call
    gives its normal, bit-identical result."""
    g = torch.Generator(device="cuda").manual_seed(43)
    S = 2.0 * torch.randn(1, 200000, 256, generator=g, device="cuda")
    P_ref, lu_ref, lv_ref = fg.focus_sinkhorn(S, 1.0, 3)
    torch.cuda.synchronize()
    assert fg.focus_get_device_status(reset=True) == 0
    fg.focus_set_wait_limit(1)
    try:
        fg.focus_sinkhorn(S, 1.0, 3)
        st = fg.focus_get_device_status(reset=True)
    finally:
        fg.focus_set_wait_limit(0)
    assert st == TIMEOUT
    P, lu, lv = fg.focus_sinkhorn(S, 1.0, 3)
    assert fg.focus_get_device_status(reset=True) == 0
    assert torch.equal(P, P_ref) and torch.equal(lu, lu_ref) and torch.equal(lv, lv_ref)
