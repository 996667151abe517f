"""focus_bucket_static: the bucketing entry point for callers that cannot
allocate device memory (for example code running inside another allocator's
callback, or an engine that has reserved the device's memory and forbids
cudaMalloc while it runs).  Instead of a caller workspace it uses a fixed
scratch array inside the library.

Checked through the C ABI against focus_bucket, which takes a workspace: two
calls in a row with different shapes, so the second call runs on the scratch
contents the first one left behind.  Bucketing is integer work, so the
results must be identical.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import learned_group_sparse_gb300 as fg
from learned_group_sparse_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_dev):
    build.build()
    fg.library()
    yield
    assert fg.focus_get_device_status(reset=True) == 0


def _ids(B, n, K, topk, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    r = torch.rand(B * n, K, generator=g, device="cuda")
    return torch.topk(r, topk, dim=1).indices.to(torch.int32).view(B, n, topk).contiguous()


def _call_static(ids_ptr, B, n, K, topk, off, pos, inv):
    st = fg.library().focus_bucket_static(
        ctypes.c_void_p(ids_ptr), B, n, K, topk, ctypes.c_void_p(off.data_ptr()),
        ctypes.c_void_p(pos.data_ptr()), ctypes.c_void_p(inv.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, fg.focus_status_string(st)


def _outputs(B, n, K, topk):
    return (torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, max(n, 1) * topk), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, max(n, 1), topk), -7, dtype=torch.int32, device="cuda"))


def test_static_scratch_matches_workspace_path_twice():
    for B, n, K, topk, seed in ((2, 50000, 256, 2, 1), (1, 30001, 64, 4, 2)):
        ids = _ids(B, n, K, topk, seed)
        off, pos, inv = _outputs(B, n, K, topk)
        _call_static(ids.data_ptr(), B, n, K, topk, off, pos, inv)
        want = fg.focus_bucket(ids, K)
        torch.cuda.synchronize()
        for a, b in zip((off, pos, inv), want):
            assert torch.equal(a, b)


def test_static_call_allocates_nothing():
    """With the outputs already allocated, a call changes neither torch's
    allocation count nor the device's free memory (the first call may load
    the library's module and its fixed array, so the check is on a repeat)."""
    B, n, K, topk = 1, 20000, 128, 2
    ids = _ids(B, n, K, topk, 3)
    off, pos, inv = _outputs(B, n, K, topk)
    _call_static(ids.data_ptr(), B, n, K, topk, off, pos, inv)
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    _call_static(ids.data_ptr(), B, n, K, topk, off, pos, inv)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    want = fg.focus_bucket(ids, K)
    torch.cuda.synchronize()
    for a, b in zip((off, pos, inv), want):
        assert torch.equal(a, b)


def test_static_empty_sequence_zeroes_offsets():
    """n = 0: no memberships, so every group offset is zero (the offsets are
    written even though nothing is scattered)."""
    B, K, topk = 2, 16, 2
    off, pos, inv = _outputs(B, 0, K, topk)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")   # never read when n = 0
    _call_static(dummy.data_ptr(), B, 0, K, topk, off, pos, inv)
    torch.cuda.synchronize()
    assert torch.equal(off, torch.zeros_like(off))


def test_static_rejects_problems_beyond_its_scratch():
    # K = 1024 and 8M (token, slot) entries need ~8 MiB x 4 of chunk counts
    need = fg.focus_bucket_workspace_size(4, 1 << 20, 1024, 8)
    assert need > (16 << 20)
    P = ctypes.c_void_p(0x10000)
    assert fg.library().focus_bucket_static(P, 4, 1 << 20, 1024, 8, P, P, P, None) == 2
