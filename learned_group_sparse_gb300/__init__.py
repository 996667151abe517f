"""Focus attention inference path for GB300 (sm_103a).

Focus (arXiv 2604.03260, "Why Attend to Everything? Focus is the Key")
scores a causal token pair (i, j) only if the tokens lie within a local
window or share one of their top-k learned centroid groups.  The work runs
in the CUDA library ``libfocus_gb300.so`` (C ABI in ``include/focus.h``);
this module is a thin ctypes binding with the same entry-point names.  It
only marshals arguments: torch provides device memory and the current
stream.  It fails loudly if the library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "FocusError", "library", "library_path",
    "focus_assign", "focus_assign_workspace_size", "focus_bucket", "focus_attention_fwd", "focus_attention_fwd_counted",
    "focus_prefill", "focus_dense_causal_fwd", "focus_count_pairs",
    "focus_bucket_workspace_size", "focus_attention_workspace_size",
    "focus_prefill_workspace_size", "focus_get_device_status", "focus_set_wait_limit",
    "focus_last_launch_count",
    "focus_status_string", "focus_version", "focus_profile_enable", "focus_profile_read",
    "focus_decode_workspace_size", "focus_decode_lists_init", "focus_decode_fwd",
    "focus_sinkhorn_workspace_size", "focus_sinkhorn",
    "focus_gated_workspace_size", "focus_gated_attention_fwd", "focus_gated_attention_bwd",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_build", "libfocus_gb300.so")
_lock = threading.Lock()
_lib = None

_STATUS = {0: "FOCUS_OK", 1: "FOCUS_ERR_INVALID_ARG", 2: "FOCUS_ERR_UNSUPPORTED",
           3: "FOCUS_ERR_WORKSPACE", 4: "FOCUS_ERR_CUDA", 5: "FOCUS_ERR_TIMEOUT",
           6: "FOCUS_ERR_CAPACITY"}


class FocusError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}")
        self.status = status


def library() -> ctypes.CDLL:
    """Loads libfocus_gb300.so (built by ``learned_group_sparse_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise FocusError("load libfocus_gb300.so (run the build first)", -1)
            lib = ctypes.CDLL(library_path)
            vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            sig = {
                "focus_status_string": ([i32], ctypes.c_char_p),
                "focus_version": ([], ctypes.c_char_p),
                "focus_assign_workspace_size": ([i32] * 6, sz),
                "focus_assign": ([vp, vp, vp] + [i32] * 6 + [vp, vp, vp, sz, vp], i32),
                "focus_bucket_workspace_size": ([i32, i32, i32, i32], sz),
                "focus_bucket": ([vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp], i32),
                "focus_attention_workspace_size": ([i32] * 7, sz),
                "focus_attention_fwd": ([vp, vp, vp] + [i32] * 6 + [f32, vp, vp, vp, vp, i32,
                                        i32, vp, vp, vp, sz, vp], i32),
                "focus_attention_fwd_counted": ([vp, vp, vp] + [i32] * 6 + [f32, vp, vp, vp, vp,
                                                i32, i32, vp, vp, vp, sz, vp, vp], i32),
                "focus_prefill_workspace_size": ([i32] * 10, sz),
                "focus_prefill": ([vp] * 6 + [i32] * 10 + [f32, vp, vp, vp, vp, sz, i32, vp],
                                  i32),
                "focus_dense_causal_fwd": ([vp, vp, vp] + [i32] * 5 + [f32, vp, vp, vp], i32),
                "focus_count_pairs": ([vp] * 4 + [i32] * 5 + [vp, vp, vp], i32),
                "focus_get_device_status": ([i32], i32),
                "focus_set_wait_limit": ([ctypes.c_ulonglong], i32),
                "focus_last_launch_count": ([], i32),
                "focus_bucket_static": ([vp, i32, i32, i32, i32, vp, vp, vp, vp], i32),
                "focus_decode_workspace_size": ([i32] * 4, sz),
                "focus_sinkhorn_workspace_size": ([i32] * 3, sz),
                "focus_gated_workspace_size": ([i32] * 5, sz),
                "focus_gated_attention_fwd": ([vp] * 4 + [i32] * 7 + [f32, f32, vp, vp, vp, sz,
                                              vp], i32),
                "focus_gated_attention_bwd": ([vp] * 7 + [i32] * 7 + [f32, f32] + [vp] * 6 +
                                              [sz, vp], i32),
                "focus_sinkhorn": ([vp, i32, i32, i32, f32, i32, vp, vp, vp, vp, sz, vp], i32),
                "focus_decode_lists_init": ([vp, vp] + [i32] * 5 + [vp, vp, vp], i32),
                "focus_decode_fwd": ([vp] * 4 + [i32] * 7 + [f32, i32, i32, vp, vp, i32, vp, vp,
                                     vp, sz, vp], i32),
                "focus_profile_enable": ([i32], None),
                "focus_trace_attention": ([vp, vp, vp], None),
                "focus_trace_gated": ([vp, vp, i32], None),
                "focus_profile_read": ([vp, i32, vp, vp, i32], i32),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _check(fn, status):
    if status != 0:
        raise FocusError(fn, status)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t=None):
    dev = t.device if t is not None and t.is_cuda else None
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t, name, dtype, dims=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def focus_status_string(status: int) -> str:
    return library().focus_status_string(status).decode()


def focus_version() -> str:
    return library().focus_version().decode()


def focus_last_launch_count() -> int:
    return int(library().focus_last_launch_count())


def focus_get_device_status(reset: bool = False) -> int:
    return int(library().focus_get_device_status(1 if reset else 0))


def focus_set_wait_limit(ns: int = 0) -> None:
    """Limit in ns of the bounded device-side waits of the launches that
    follow (0: the default, 2 s); the attention kernels keep the default.
    A testing aid for the timeout path."""
    _check("focus_set_wait_limit", library().focus_set_wait_limit(int(ns)))


def focus_profile_enable(enable: bool = True) -> None:
    library().focus_profile_enable(1 if enable else 0)


def focus_profile_read(max_entries: int = 64) -> dict:
    """{kernel name: (total ms, launches)} since the last read."""
    stride = 64
    names = ctypes.create_string_buffer(stride * max_entries)
    ms = (ctypes.c_double * max_entries)()
    cnt = (ctypes.c_int * max_entries)()
    k = library().focus_profile_read(names, stride, ms, cnt, max_entries)
    if k < 0:
        raise FocusError("focus_profile_read", 4)
    out = {}
    for i in range(k):
        nm = names.raw[i * stride:(i + 1) * stride].split(b"\0", 1)[0].decode()
        out[nm] = (float(ms[i]), int(cnt[i]))
    return out


def focus_trace_gated(query_buf=None, key_buf=None, max_ctas=0) -> None:
    """Sets (or with None / 0 clears) the per-CTA wait-trace buffers of the
    gated backward, int64 CUDA tensors of at least 32 x max_ctas entries."""
    library().focus_trace_gated(_p(query_buf), _p(key_buf), int(max_ctas))


def focus_trace_attention(group_buf=None, window_buf=None, dense_buf=None) -> None:
    """Sets (or with None clears) the per-CTA wait-trace buffers, int64 CUDA
    tensors of >= 32 x SM-count entries, of the group/window/dense kernels."""
    library().focus_trace_attention(_p(group_buf), _p(window_buf), _p(dense_buf))


def focus_assign_workspace_size(B, n, hidden, dg, K, topk) -> int:
    return int(library().focus_assign_workspace_size(B, n, hidden, dg, K, topk))


def focus_assign(X, Wg, C, topk, ids=None, margin=None, with_margin=True, ws=None):
    """X [B, n, hidden] bf16, Wg [hidden, d_g] fp32, C [K, d_g] fp32 ->
    (ids [B, n, topk] int32, margin [B, n] fp32 or None)."""
    _need(X, "X", torch.bfloat16, 3)
    _need(Wg, "Wg", torch.float32, 2)
    _need(C, "C", torch.float32, 2)
    B, n, hidden = X.shape
    K, dg = C.shape
    if ids is None:
        ids = torch.empty(B, n, topk, dtype=torch.int32, device=X.device)
    if margin is None and with_margin:
        margin = torch.empty(B, n, dtype=torch.float32, device=X.device)
    need = focus_assign_workspace_size(B, n, hidden, dg, K, topk)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=X.device)
    _check("focus_assign", library().focus_assign(
        _p(X), _p(Wg), _p(C), B, n, hidden, dg, K, topk, _p(ids), _p(margin), _p(ws),
        0 if ws is None else ws.numel(), _stream(X)))
    return ids, margin


def focus_bucket_workspace_size(B, n, K, topk) -> int:
    return int(library().focus_bucket_workspace_size(B, n, K, topk))


def focus_bucket(ids, num_groups, offsets=None, pos=None, inv=None, ws=None):
    """ids [B, n, topk] int32 -> (offsets [B, K+1], pos [B, n*topk], inv [B, n, topk])."""
    _need(ids, "ids", torch.int32, 3)
    B, n, topk = ids.shape
    dev = ids.device
    if offsets is None:
        offsets = torch.empty(B, num_groups + 1, dtype=torch.int32, device=dev)
    if pos is None:
        pos = torch.empty(B, n * topk, dtype=torch.int32, device=dev)
    if inv is None:
        inv = torch.empty(B, n, topk, dtype=torch.int32, device=dev)
    need = focus_bucket_workspace_size(B, n, num_groups, topk)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    _check("focus_bucket", library().focus_bucket(
        _p(ids), B, n, num_groups, topk, _p(offsets), _p(pos), _p(inv), _p(ws), ws.numel(),
        _stream(ids)))
    return offsets, pos, inv


def focus_bucket_static(ids, num_groups, offsets=None, pos=None, inv=None):
    """focus_bucket for callers that cannot allocate device memory: the
    library's own fixed scratch array replaces the workspace (16 MiB limit;
    calls overlapping on the GPU race).  Output buffers may be passed in so
    that nothing at all is allocated."""
    _need(ids, "ids", torch.int32, 3)
    B, n, topk = ids.shape
    dev = ids.device
    if offsets is None:
        offsets = torch.empty(B, num_groups + 1, dtype=torch.int32, device=dev)
    if pos is None:
        pos = torch.empty(B, n * topk, dtype=torch.int32, device=dev)
    if inv is None:
        inv = torch.empty(B, n, topk, dtype=torch.int32, device=dev)
    _check("focus_bucket_static", library().focus_bucket_static(
        _p(ids), B, n, num_groups, topk, _p(offsets), _p(pos), _p(inv), _stream(ids)))
    return offsets, pos, inv


def focus_attention_workspace_size(B, n, Hq, Hkv, d, K, topk) -> int:
    return int(library().focus_attention_workspace_size(B, n, Hq, Hkv, d, K, topk))


def _attn_prep(Q, K, V, ids, offsets, pos, inv, O, lse, ws, num_groups, with_lse):
    for t, name in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, name, torch.bfloat16, 4)
    for t, name in ((ids, "ids"), (offsets, "offsets"), (pos, "pos"), (inv, "inv")):
        _need(t, name, torch.int32)
    B, n, Hq, d = Q.shape
    Hkv = K.shape[2]
    topk = ids.shape[-1]
    if O is None:
        O = torch.empty_like(Q)
    if lse is None and with_lse:
        lse = torch.empty(B, Hq, n, dtype=torch.float32, device=Q.device)
    need = focus_attention_workspace_size(B, n, Hq, Hkv, d, num_groups, topk)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=Q.device)
    return B, n, Hq, Hkv, d, topk, O, lse, ws


def focus_attention_fwd(Q, K, V, window, ids, offsets, pos, inv, num_groups, scale=0.0,
                        O=None, lse=None, ws=None, with_lse=True):
    """Focus attention.  Q [B, n, Hq, d], K/V [B, n, Hkv, d] bf16 -> (O, lse [B, Hq, n])."""
    B, n, Hq, Hkv, d, topk, O, lse, ws = _attn_prep(Q, K, V, ids, offsets, pos, inv, O, lse, ws,
                                                    num_groups, with_lse)
    _check("focus_attention_fwd", library().focus_attention_fwd(
        _p(Q), _p(K), _p(V), B, n, Hq, Hkv, d, int(window), float(scale), _p(ids), _p(offsets),
        _p(pos), _p(inv), num_groups, topk, _p(O), _p(lse), _p(ws), ws.numel(), _stream(Q)))
    return O, lse


def focus_attention_fwd_counted(Q, K, V, window, ids, offsets, pos, inv, num_groups, scale=0.0,
                                O=None, lse=None, ws=None):
    """As focus_attention_fwd, plus the number of pairs scored per query
    (head 0), int32 [B, n]."""
    B, n, Hq, Hkv, d, topk, O, lse, ws = _attn_prep(Q, K, V, ids, offsets, pos, inv, O, lse, ws,
                                                    num_groups, True)
    cnt = torch.zeros(B, n, dtype=torch.int32, device=Q.device)
    _check("focus_attention_fwd_counted", library().focus_attention_fwd_counted(
        _p(Q), _p(K), _p(V), B, n, Hq, Hkv, d, int(window), float(scale), _p(ids), _p(offsets),
        _p(pos), _p(inv), num_groups, topk, _p(O), _p(lse), _p(ws), ws.numel(), _p(cnt),
        _stream(Q)))
    return O, lse, cnt


def focus_prefill_workspace_size(B, n, hidden, Hq, Hkv, d, dg, K, topk, io_on_host) -> int:
    return int(library().focus_prefill_workspace_size(B, n, hidden, Hq, Hkv, d, dg, K, topk,
                                                      1 if io_on_host else 0))


def focus_prefill(X, Wg, C, Q, K, V, topk, window, scale=0.0, O=None, lse=None, ids_out=None,
                  ws=None, stream=None):
    """The whole path in one call.  Tensors all on the GPU, or all on the host
    (pinned) with O/lse host outputs; the copies then run inside the call."""
    host = not Q.is_cuda
    B, n, hidden = X.shape
    Hq, d = Q.shape[2], Q.shape[3]
    Hkv = K.shape[2]
    Kg, dg = C.shape
    for t, name, dt in ((X, "X", torch.bfloat16), (Wg, "Wg", torch.float32),
                        (C, "C", torch.float32), (Q, "Q", torch.bfloat16),
                        (K, "K", torch.bfloat16), (V, "V", torch.bfloat16)):
        _need(t, name, dt, cuda=not host)
    if O is None:
        O = torch.empty(B, n, Hq, d, dtype=torch.bfloat16, device=Q.device,
                        pin_memory=host)
    if ws is None:
        need = focus_prefill_workspace_size(B, n, hidden, Hq, Hkv, d, dg, Kg, topk, host)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = ctypes.c_void_p(stream) if stream is not None else _stream(ws)
    _check("focus_prefill", library().focus_prefill(
        _p(X), _p(Wg), _p(C), _p(Q), _p(K), _p(V), B, n, hidden, Hq, Hkv, d, dg, Kg, topk,
        int(window), float(scale), _p(O), _p(lse), _p(ids_out), _p(ws), ws.numel(),
        1 if host else 0, s))
    return O, lse


def focus_gated_workspace_size(B, n, Hq, Hkv, Kg) -> int:
    return int(library().focus_gated_workspace_size(B, n, Hq, Hkv, Kg))


def _gated_common(Q, K, V, G):
    _need(Q, "Q", torch.bfloat16, 4)
    _need(K, "K", torch.bfloat16, 4)
    _need(V, "V", torch.bfloat16, 4)
    _need(G, "G", torch.float32, 3)
    B, n, Hq, d = Q.shape
    return B, n, Hq, K.shape[2], d, G.shape[2]


def focus_gated_attention_fwd(Q, K, V, G, window, lam, scale=0.0, O=None, lse=None, ws=None):
    """Soft-gated causal attention of training: Q [B, n, Hq, d], K/V
    [B, n, Hkv, d] bf16, G [B, n, Kg] fp32 soft assignments -> (O bf16,
    lse [B, Hq, n] fp32)."""
    B, n, Hq, Hkv, d, Kg = _gated_common(Q, K, V, G)
    if O is None:
        O = torch.empty_like(Q)
    if lse is None:
        lse = torch.empty(B, Hq, n, dtype=torch.float32, device=Q.device)
    if ws is None:
        ws = torch.empty(max(1, focus_gated_workspace_size(B, n, Hq, Hkv, Kg)), dtype=torch.uint8,
                         device=Q.device)
    _check("focus_gated_attention_fwd", library().focus_gated_attention_fwd(
        _p(Q), _p(K), _p(V), _p(G), B, n, Hq, Hkv, d, Kg, int(window), float(lam), float(scale),
        _p(O), _p(lse), _p(ws), ws.numel(), _stream(Q)))
    return O, lse


def focus_gated_attention_bwd(Q, K, V, G, O, lse, dO, window, lam, scale=0.0, ws=None,
                              out=None):
    """Gradients of the soft-gated attention -> (dQ, dK, dV, dG, dlambda),
    fp32 tensors (dlambda of one element).  out: optional tuple of the five
    output tensors to fill."""
    B, n, Hq, Hkv, d, Kg = _gated_common(Q, K, V, G)
    _need(O, "O", torch.bfloat16, 4)
    _need(dO, "dO", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    dev = Q.device
    if out is None:
        out = (torch.empty(B, n, Hq, d, dtype=torch.float32, device=dev),
               torch.empty(B, n, Hkv, d, dtype=torch.float32, device=dev),
               torch.empty(B, n, Hkv, d, dtype=torch.float32, device=dev),
               torch.empty(B, n, Kg, dtype=torch.float32, device=dev),
               torch.empty(1, dtype=torch.float32, device=dev))
    if ws is None:
        ws = torch.empty(max(1, focus_gated_workspace_size(B, n, Hq, Hkv, Kg)), dtype=torch.uint8,
                         device=dev)
    dQ, dK, dV, dG, dl = out
    _check("focus_gated_attention_bwd", library().focus_gated_attention_bwd(
        _p(Q), _p(K), _p(V), _p(G), _p(O), _p(lse), _p(dO), B, n, Hq, Hkv, d, Kg, int(window),
        float(lam), float(scale), _p(dQ), _p(dK), _p(dV), _p(dG), _p(dl), _p(ws), ws.numel(),
        _stream(Q)))
    return dQ, dK, dV, dG, dl


def focus_sinkhorn_workspace_size(B, n, K) -> int:
    return int(library().focus_sinkhorn_workspace_size(B, n, K))


def focus_sinkhorn(S, tau=1.0, iters=3, P=None, log_u=None, log_v=None, ws=None, want_p=True):
    """Sinkhorn normalisation of affinities S [B, n, K] fp32 (rows to mass 1,
    groups to mass n / K, `iters` rounds) -> (P [B, n, K] or None,
    log_u [B, n], log_v [B, K]), fp32."""
    _need(S, "S", torch.float32, 3)
    B, n, K = S.shape
    dev = S.device
    if P is None and want_p:
        P = torch.empty(B, n, K, dtype=torch.float32, device=dev)
    if log_u is None:
        log_u = torch.empty(B, n, dtype=torch.float32, device=dev)
    if log_v is None:
        log_v = torch.empty(B, K, dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(max(1, focus_sinkhorn_workspace_size(B, n, K)), dtype=torch.uint8,
                         device=dev)
    _check("focus_sinkhorn", library().focus_sinkhorn(
        _p(S), B, n, K, float(tau), int(iters), _p(P), _p(log_u), _p(log_v), _p(ws), ws.numel(),
        _stream(S)))
    return P, log_u, log_v


def focus_decode_workspace_size(B, Hq, Hkv, d) -> int:
    return int(library().focus_decode_workspace_size(B, Hq, Hkv, d))


def focus_decode_lists_init(offsets, pos, num_groups, topk, cap, glen=None, gpos=None):
    """Group lists with room for `cap` members each, from a prefix's bucketing
    (offsets [B, K+1], pos [B, n*topk] of focus_bucket) -> (glen [B, K],
    gpos [B, K, cap]) int32."""
    _need(offsets, "offsets", torch.int32, 2)
    _need(pos, "pos", torch.int32, 2)
    B = offsets.shape[0]
    n = pos.shape[1] // topk
    dev = offsets.device
    if glen is None:
        glen = torch.empty(B, num_groups, dtype=torch.int32, device=dev)
    if gpos is None:
        gpos = torch.empty(B, num_groups, cap, dtype=torch.int32, device=dev)
    # a prefix of no tokens has an empty pos tensor: pass any valid pointer
    pos_p = _p(pos) if pos.numel() else _p(glen)
    _check("focus_decode_lists_init", library().focus_decode_lists_init(
        _p(offsets), pos_p, B, n, num_groups, topk, cap, _p(glen), _p(gpos), _stream(offsets)))
    return glen, gpos


def focus_decode_fwd(q, Kc, Vc, ids, L, window, glen, gpos, num_groups, scale=0.0, O=None,
                     lse=None, ws=None, with_lse=True):
    """One new token per sequence (position L - 1 of the cache): appends it to
    its groups' lists (glen/gpos, in place) and attends over its allowed keys.
    q [B, Hq, d], Kc/Vc [B, Lmax, Hkv, d] bf16, ids [B, Lmax, topk] int32 ->
    (O [B, Hq, d] bf16, lse [B, Hq] fp32 or None)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(Kc, "Kc", torch.bfloat16, 4)
    _need(Vc, "Vc", torch.bfloat16, 4)
    _need(ids, "ids", torch.int32, 3)
    _need(glen, "glen", torch.int32, 2)
    _need(gpos, "gpos", torch.int32, 3)
    B, Hq, d = q.shape
    Lmax, Hkv = Kc.shape[1], Kc.shape[2]
    topk = ids.shape[-1]
    cap = gpos.shape[-1]
    if O is None:
        O = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    need = focus_decode_workspace_size(B, Hq, Hkv, d)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check("focus_decode_fwd", library().focus_decode_fwd(
        _p(q), _p(Kc), _p(Vc), _p(ids), B, int(L), Lmax, Hq, Hkv, d, int(window), float(scale),
        num_groups, topk, _p(glen), _p(gpos), cap, _p(O), _p(lse), _p(ws), ws.numel(),
        _stream(q)))
    return O, lse


def focus_dense_causal_fwd(Q, K, V, scale=0.0, O=None, lse=None, with_lse=False):
    """Plain causal attention with the same tcgen05 mainloop."""
    for t, name in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, name, torch.bfloat16, 4)
    B, n, Hq, d = Q.shape
    Hkv = K.shape[2]
    if O is None:
        O = torch.empty_like(Q)
    if lse is None and with_lse:
        lse = torch.empty(B, Hq, n, dtype=torch.float32, device=Q.device)
    _check("focus_dense_causal_fwd", library().focus_dense_causal_fwd(
        _p(Q), _p(K), _p(V), B, n, Hq, Hkv, d, float(scale), _p(O), _p(lse), _stream(Q)))
    return O, lse


def focus_count_pairs(ids, offsets, pos, inv, num_groups, window, per_query=True):
    """-> (per_query int64 [B, n] or None, totals int64 [2] on device):
    totals[0] = sum |A_i|, totals[1] = pairs sharing a group."""
    B, n, topk = ids.shape
    per = torch.empty(B, n, dtype=torch.int64, device=ids.device) if per_query else None
    tot = torch.empty(2, dtype=torch.int64, device=ids.device)
    _check("focus_count_pairs", library().focus_count_pairs(
        _p(ids), _p(offsets), _p(pos), _p(inv), B, n, num_groups, topk, int(window), _p(per),
        _p(tot), _stream(ids)))
    return per, tot
