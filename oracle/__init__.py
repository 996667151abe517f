"""Focus attention oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU implementation of the Focus inference path written from
the web summaries of arXiv 2604.03260 ("Why Attend to Everything? Focus is
the Key"), used to check the CUDA library.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with ``learned_group_sparse_gb300`` and
imports nothing from it.

The arithmetic lives in ``focus_oracle.c`` (plain C, OpenMP over query rows,
double accumulation); this module only compiles it and marshals numpy
arrays.  Function-by-function sources:

* :func:`assign` -- token grouping and hard top-k membership
  (gist.science/zh technical summary 2.1.1 and 2.1.3; gist.science/nl
  Kerncomponenten 1 and 4).
* :func:`bucket` -- per-group member lists in ascending token order (implied
  by "within-group causal attention", gist.science/zh 2.1.3).
* :func:`attention` -- exact softmax over the allowed pairs: local window or
  a shared group, causal (gist.science/nl Kerncomponenten 3; gist.science/zh
  2.1.2 and 2.1.3).
* :func:`count_pairs` -- |A_i| by enumeration of the same rule.
* :func:`gated_fwd`, :func:`gated_bwd` -- the soft-gated attention of
  training over all causal pairs and its gradients (gist.science/zh 2.1.2;
  gist.science/nl Kerncomponent 4).
* :func:`sinkhorn` -- Sinkhorn normalisation of the training-time
  token-group affinities (gist.science/nl Kerncomponenten 2; gist.science/zh
  2.1.1): rows to mass 1, groups to equal mass n / K.

Parity status: every function is pinned by ``tests/test_oracle_pins.py``
(brute force on tiny inputs, closed forms, special cases that reduce to
library routines); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "focus_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_focus.so")
_lock = threading.Lock()
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile focus_oracle.c into a shared library (gcc, OpenMP if present)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.oracle_assign.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, vp, vp, vp]
            lib.oracle_bucket.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
            lib.oracle_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                                             vp, i32, vp, i64, i32, vp, vp]
            lib.oracle_count_pairs.argtypes = [vp, i32, i32, i32, i32, vp, i64, vp, _I64P]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_sinkhorn.argtypes = [vp, i32, i32, i32, ctypes.c_double, i32, vp, vp, vp]
            f64 = ctypes.c_double
            lib.oracle_gated_fwd.argtypes = [vp, vp, vp, vp] + [i32] * 7 + [f64, f64, vp, vp]
            lib.oracle_gated_bwd.argtypes = [vp] * 5 + [i32] * 7 + [f64, f64] + [vp] * 6
            for f in (lib.oracle_assign, lib.oracle_bucket, lib.oracle_attention,
                      lib.oracle_count_pairs, lib.oracle_num_threads, lib.oracle_sinkhorn,
                      lib.oracle_gated_fwd, lib.oracle_gated_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a):
    """bf16 data as a contiguous uint16 array of raw bit patterns."""
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def assign(X_bits, Wg, C, topk):
    """Hard top-k group membership.

    X_bits: [..., hidden] uint16 (bf16 bits); Wg: [hidden, d_g] float32;
    C: [K, d_g] float32.  Returns (ids [..., topk] int32 by descending score,
    ties to the lower id; margin [...] float32; scores [..., K] float32).
    """
    X = _bits16(X_bits)
    lead = X.shape[:-1]
    hidden = X.shape[-1]
    Wg = np.ascontiguousarray(Wg, dtype=np.float32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    K, dg = C.shape
    assert Wg.shape == (hidden, dg)
    ntok = int(np.prod(lead)) if lead else 1
    ids = np.empty((ntok, topk), np.int32)
    margin = np.empty((ntok,), np.float32)
    scores = np.empty((ntok, K), np.float32)
    rc = _load().oracle_assign(_ptr(X), _ptr(Wg), _ptr(C), ntok, hidden, dg, K, topk,
                               _ptr(ids), _ptr(margin), _ptr(scores))
    if rc:
        raise ValueError("oracle_assign: invalid arguments")
    return ids.reshape(*lead, topk), margin.reshape(lead), scores.reshape(*lead, K)


def bucket(ids, K):
    """Group lists.  ids [B, n, topk] int32 -> (offsets [B, K+1],
    pos [B, n*topk], inv [B, n, topk]), all int32, per-batch indices."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    B, n, topk = ids.shape
    offsets = np.empty((B, K + 1), np.int32)
    pos = np.empty((B, n * topk), np.int32)
    inv = np.empty((B, n, topk), np.int32)
    rc = _load().oracle_bucket(_ptr(ids), B, n, K, topk, _ptr(offsets), _ptr(pos), _ptr(inv))
    if rc:
        raise ValueError("oracle_bucket: invalid arguments")
    return offsets, pos, inv


def attention(Q_bits, K_bits, V_bits, ids, window, scale=0.0, rows=None):
    """Exact masked-softmax attention over the allowed pairs.

    Q_bits [B, n, Hq, d], K_bits/V_bits [B, n, Hkv, d] uint16 (bf16 bits);
    ids [B, n, topk] int32.  rows: optional 1-D int64 array of flattened query
    indices b*n + i; then Q_bits may instead hold just those rows,
    [len(rows), Hq, d].  Returns (O [rows, Hq, d] float32, LSE [rows, Hq]
    float32, natural log); with rows=None the leading shape is [B, n].
    """
    Q, Kt, V = _bits16(Q_bits), _bits16(K_bits), _bits16(V_bits)
    B, n, Hkv, d = Kt.shape
    q_rows_only = Q.ndim == 3
    Hq = Q.shape[-2]
    if q_rows_only:
        assert rows is not None and Q.shape[0] == len(rows)
    else:
        assert Q.shape == (B, n, Hq, d)
    assert V.shape == Kt.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    topk = ids.shape[-1]
    assert ids.shape == (B, n, topk)
    if rows is None:
        nrows, rows_arr = B * n, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.shape[0]
    O = np.empty((nrows, Hq, d), np.float32)
    L = np.empty((nrows, Hq), np.float32)
    rc = _load().oracle_attention(_ptr(Q), _ptr(Kt), _ptr(V), B, n, Hq, Hkv, d, int(window),
                                  float(scale), _ptr(ids), topk, _ptr(rows_arr), nrows,
                                  1 if q_rows_only else 0, _ptr(O), _ptr(L))
    if rc:
        raise ValueError("oracle_attention: invalid arguments")
    if rows is None:
        return O.reshape(B, n, Hq, d), L.reshape(B, n, Hq)
    return O, L


def count_pairs(ids, window, rows=None):
    """Allowed keys per query.  ids [B, n, topk] -> (per_query [B, n] int64,
    total).  rows: optional 1-D int64 array of flattened query indices b*n + i;
    then per_query is [len(rows)] and total sums over those rows only."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    B, n, topk = ids.shape
    if rows is None:
        rows_arr, nrows = None, B * n
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.shape[0]
    per = np.empty((nrows,), np.int64)
    tot = ctypes.c_int64(0)
    rc = _load().oracle_count_pairs(_ptr(ids), B, n, topk, int(window), _ptr(rows_arr), nrows,
                                    _ptr(per), ctypes.byref(tot))
    if rc:
        raise ValueError("oracle_count_pairs: invalid arguments")
    return (per.reshape(B, n) if rows is None else per), int(tot.value)


def sinkhorn(S, tau=1.0, iters=3, want_p=True):
    """Sinkhorn-Knopp scaling of exp(S / tau), S [B, n, K] float32: `iters`
    rounds of (rows to mass 1, then groups to mass n / K), from v = 1.
    Returns (P [B, n, K] or None, log_u [B, n], log_v [B, K]), float64."""
    S = np.ascontiguousarray(S, dtype=np.float32)
    B, n, K = S.shape
    P = np.empty((B, n, K), np.float64) if want_p else None
    lu = np.empty((B, n), np.float64)
    lv = np.empty((B, K), np.float64)
    rc = _load().oracle_sinkhorn(_ptr(S), B, n, K, float(tau), int(iters), _ptr(P), _ptr(lu),
                                 _ptr(lv))
    if rc:
        raise ValueError("oracle_sinkhorn: invalid arguments")
    return P, lu, lv


def _gated_shapes(Q_bits, K_bits, V_bits, G):
    Q, K, V = _bits16(Q_bits), _bits16(K_bits), _bits16(V_bits)
    G = np.ascontiguousarray(G, dtype=np.float32)
    B, n, Hq, d = Q.shape
    Hkv = K.shape[2]
    return Q, K, V, G, B, n, Hq, Hkv, d, G.shape[2]


def gated_fwd(Q_bits, K_bits, V_bits, G, window, lam, scale=0.0):
    """Soft-gated causal attention: Q [B, n, Hq, d], K/V [B, n, Hkv, d] as bf16
    bit patterns, G [B, n, Kg] float32 -> (O [B, n, Hq, d], LSE [B, Hq, n]),
    float64."""
    Q, K, V, G, B, n, Hq, Hkv, d, Kg = _gated_shapes(Q_bits, K_bits, V_bits, G)
    O = np.empty((B, n, Hq, d), np.float64)
    L = np.empty((B, Hq, n), np.float64)
    rc = _load().oracle_gated_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(G), B, n, Hq, Hkv, d, Kg,
                                  int(window), float(lam), float(scale), _ptr(O), _ptr(L))
    if rc:
        raise ValueError("oracle_gated_fwd: invalid arguments")
    return O, L


def gated_bwd(Q_bits, K_bits, V_bits, G, dO, window, lam, scale=0.0, with_abs=False):
    """Gradients of sum(O * dO) for the soft-gated attention -> (dQ, dK, dV,
    dG, dlambda), float64; with_abs appends the sum of the magnitudes of
    dlambda's per-pair terms."""
    Q, K, V, G, B, n, Hq, Hkv, d, Kg = _gated_shapes(Q_bits, K_bits, V_bits, G)
    dO = np.ascontiguousarray(dO, dtype=np.float32)
    dQ = np.empty((B, n, Hq, d), np.float64)
    dK = np.empty((B, n, Hkv, d), np.float64)
    dV = np.empty((B, n, Hkv, d), np.float64)
    dG = np.empty((B, n, Kg), np.float64)
    dl = ctypes.c_double(0.0)
    dl_abs = ctypes.c_double(0.0)
    rc = _load().oracle_gated_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(G), _ptr(dO), B, n, Hq, Hkv,
                                  d, Kg, int(window), float(lam), float(scale), _ptr(dQ),
                                  _ptr(dK), _ptr(dV), _ptr(dG), ctypes.byref(dl),
                                  ctypes.byref(dl_abs))
    if rc:
        raise ValueError("oracle_gated_bwd: invalid arguments")
    if with_abs:
        return dQ, dK, dV, dG, float(dl.value), float(dl_abs.value)
    return dQ, dK, dV, dG, float(dl.value)
