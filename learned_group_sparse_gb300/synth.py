"""Seeded synthetic inputs for the Focus inference path.

This module holds no arithmetic of the method: it only draws inputs with the
shapes and structure of the five workloads below, so that the CUDA library
and the CPU oracle can be fed identical bits.  Randomness comes from a
``torch.Generator`` seeded with ``1000 + index`` (or an explicit seed).

The pages measure quality on PG-19 and downstream suites; those are not this
path.  The stand-ins are:

* Gaussian X (small case), or a Gaussian mixture aligned to the centroids:
  W_g gets orthonormal columns, component c has mean alpha * W_g C_c^T and
  X = mean + sigma * noise, so a token's own centroid wins its top-1 and the
  remaining choices are near-random; mixture weights uniform (balanced
  groups) or Zipf(s) (skewed groups).
* Q, K, V ~ N(0, 1) in bf16; centroids are unit-norm fp32 rows.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    n: int
    hidden: int
    Hq: int
    Hkv: int
    d: int
    K: int
    dg: int
    topk: int
    window: int
    x_kind: str = "mixture"      # "normal" | "mixture"
    zipf_s: float = 0.0          # 0: balanced mixture weights
    alpha: float = 4.0           # distance of a component mean from the origin
    sigma: float = 0.5           # mixture noise
    seed: int = 0

    @property
    def label(self) -> str:
        kv = "MHA" if self.Hq == self.Hkv else f"GQA{self.Hq}/{self.Hkv}"
        return (f"B{self.B} n{self.n} hidden{self.hidden} {kv} H{self.Hq} d{self.d} "
                f"K{self.K} d_g{self.dg} top{self.topk} w{self.window}"
                + (f" zipf{self.zipf_s}" if self.zipf_s else ""))


WORKLOADS = [
    Workload("n1k_mha12_d64_K16_top1_w64", 1, 1024, 768, 12, 12, 64, 16, 64, 1, 64,
             x_kind="normal", seed=1000),
    Workload("n8k_mha32_d128_K64_top2_w256", 1, 8192, 4096, 32, 32, 128, 64, 128, 2, 256,
             seed=1001),
    Workload("b2_n32k_gqa32x8_d128_K64_top2_w512", 2, 32768, 4096, 32, 8, 128, 64, 128, 2, 512,
             seed=1002),
    Workload("n128k_gqa32x8_d128_K128_top4_w1024_zipf", 1, 131072, 4096, 32, 8, 128, 128, 128,
             4, 1024, zipf_s=1.1, seed=1003),
    Workload("n1m_gqa32x8_d128_K256_top2_w1024", 1, 1048576, 4096, 32, 8, 128, 256, 128, 2,
             1024, seed=1004),
]


def workload(i_or_name) -> Workload:
    if isinstance(i_or_name, int):
        return WORKLOADS[i_or_name]
    for w in WORKLOADS:
        if w.name == i_or_name:
            return w
    raise KeyError(i_or_name)


def small(**kw) -> Workload:
    """A custom workload for tests (defaults: a tiny MHA case)."""
    base = dict(name="custom", B=1, n=300, hidden=64, Hq=2, Hkv=2, d=64, K=8, dg=16,
                topk=2, window=16, x_kind="mixture", seed=7)
    base.update(kw)
    return Workload(**base)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_params(w: Workload, device="cpu", gen=None):
    """W_g [hidden, d_g] fp32 and centroids C [K, d_g] fp32 (unit rows)."""
    g = gen if gen is not None else _gen(device, w.seed)
    C = torch.randn(w.K, w.dg, generator=g, device=device, dtype=torch.float32)
    C = C / C.norm(dim=1, keepdim=True)
    if w.x_kind == "normal":
        Wg = torch.randn(w.hidden, w.dg, generator=g, device=device,
                         dtype=torch.float32) / float(np.sqrt(w.hidden))
    else:
        A = torch.randn(w.hidden, w.dg, generator=g, device=device, dtype=torch.float32)
        Wg = torch.linalg.qr(A.cpu().double())[0].float().to(device)
    return Wg.contiguous(), C.contiguous()


def mixture_weights(w: Workload) -> torch.Tensor:
    if w.zipf_s:
        r = torch.arange(1, w.K + 1, dtype=torch.float64)
        p = r.pow(-w.zipf_s)
    else:
        p = torch.ones(w.K, dtype=torch.float64)
    return p / p.sum()


def make_components(w: Workload, device="cpu", gen=None):
    """Mixture component of every token, [B, n] int64."""
    g = gen if gen is not None else _gen(device, w.seed + 1)
    p = mixture_weights(w).to(device=device, dtype=torch.float32)
    return torch.multinomial(p, w.B * w.n, replacement=True, generator=g).view(w.B, w.n)


def make_x(w: Workload, Wg, C, comp, device="cpu", gen=None, chunk_rows=1 << 16):
    """Hidden states X [B, n, hidden] bf16."""
    g = gen if gen is not None else _gen(device, w.seed + 2)
    X = torch.empty(w.B * w.n, w.hidden, dtype=torch.bfloat16, device=device)
    if w.x_kind == "normal":
        for s in range(0, w.B * w.n, chunk_rows):
            e = min(s + chunk_rows, w.B * w.n)
            X[s:e] = torch.randn(e - s, w.hidden, generator=g, device=device).to(torch.bfloat16)
    else:
        means = (w.alpha * (C @ Wg.t())).to(device)          # [K, hidden]
        flat = comp.reshape(-1).to(device)
        for s in range(0, w.B * w.n, chunk_rows):
            e = min(s + chunk_rows, w.B * w.n)
            noise = torch.randn(e - s, w.hidden, generator=g, device=device)
            X[s:e] = (means[flat[s:e]] + w.sigma * noise).to(torch.bfloat16)
    return X.view(w.B, w.n, w.hidden)


def make_qkv(w: Workload, device="cpu", gen=None):
    """Q [B, n, Hq, d], K and V [B, n, Hkv, d], N(0, 1) in bf16."""
    g = gen if gen is not None else _gen(device, w.seed + 3)
    Q = torch.randn(w.B, w.n, w.Hq, w.d, generator=g, device=device, dtype=torch.bfloat16)
    K = torch.randn(w.B, w.n, w.Hkv, w.d, generator=g, device=device, dtype=torch.bfloat16)
    V = torch.randn(w.B, w.n, w.Hkv, w.d, generator=g, device=device, dtype=torch.bfloat16)
    return Q, K, V


def synthetic_ids(w: Workload, comp, device="cpu", gen=None, chunk_rows=1 << 16):
    """Group ids with the structure hard top-k assignment gives on the mixture
    inputs: the first id is the token's own component, the other topk-1 are
    distinct uniformly random groups.  [B, n, topk] int32."""
    g = gen if gen is not None else _gen(device, w.seed + 4)
    flat = comp.reshape(-1).to(device)
    out = torch.empty(flat.numel(), w.topk, dtype=torch.int32, device=device)
    for s in range(0, flat.numel(), chunk_rows):
        e = min(s + chunk_rows, flat.numel())
        r = torch.rand(e - s, w.K, generator=g, device=device)
        r.scatter_(1, flat[s:e, None], 2.0)
        out[s:e] = torch.topk(r, w.topk, dim=1).indices.to(torch.int32)
    return out.view(w.B, w.n, w.topk)


def synthetic_affinities(w: Workload, comp, boost=4.0, device="cpu", gen=None,
                         chunk_rows=1 << 16):
    """Token-group affinities with the mixture's structure, for the Sinkhorn
    normalisation: N(0, 1) everywhere plus `boost` on the token's own
    component.  [B, n, K] float32."""
    g = gen if gen is not None else _gen(device, w.seed + 5)
    flat = comp.reshape(-1).to(device)
    out = torch.empty(flat.numel(), w.K, dtype=torch.float32, device=device)
    for s in range(0, flat.numel(), chunk_rows):
        e = min(s + chunk_rows, flat.numel())
        r = torch.randn(e - s, w.K, generator=g, device=device)
        r.scatter_add_(1, flat[s:e, None], torch.full((e - s, 1), boost, device=device))
        out[s:e] = r
    return out.view(w.B, w.n, w.K)


def make_all(w: Workload, device="cpu", with_x=True):
    """Every input of one forward pass, drawn in a fixed order."""
    Wg, C = make_params(w, device)
    comp = make_components(w, device)
    X = make_x(w, Wg, C, comp, device) if with_x else None
    Q, K, V = make_qkv(w, device)
    return dict(Wg=Wg, C=C, comp=comp, X=X, Q=Q, K=K, V=V)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
