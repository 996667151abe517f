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
