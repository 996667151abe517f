"""Shared helpers of the GPU parity tests (comparison rules and row sampling)."""
import numpy as np
import torch

# Tolerances for bf16 I/O with fp32 accumulation: max-abs 1e-2, mean-abs 1e-3
# on the attention output; ids bit-exact where the top-k margin exceeds 1e-4.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 2e-3
MARGIN = 1e-4


def check_output(O_gpu, O_ref, L_gpu=None, L_ref=None, label=""):
    """O_gpu: bf16 tensor [..., d] (any device); O_ref: float32 ndarray, same shape."""
    o = O_gpu.float().cpu().numpy()
    err = np.abs(o - O_ref)
    assert np.isfinite(o).all(), f"{label}: non-finite output"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{label}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    if L_gpu is not None:
        lerr = np.abs(L_gpu.float().cpu().numpy() - L_ref)
        assert float(lerr.max()) <= LSE_ABS, f"{label}: lse max-abs {float(lerr.max()):.3e}"
    return mx, mean


def check_ids(ids_gpu, ids_ref, margin_ref):
    """ids bit-exact where the oracle's margin > 1e-4; elsewhere skipped.
    Returns the number of skipped tokens."""
    g = ids_gpu.cpu().numpy().reshape(-1, ids_ref.shape[-1])
    r = ids_ref.reshape(-1, ids_ref.shape[-1])
    m = margin_ref.reshape(-1)
    sure = m > MARGIN
    bad = np.nonzero((g != r).any(-1) & sure)[0]
    assert bad.size == 0, f"{bad.size} ids differ with margin > 1e-4, first token {bad[:5]}"
    return int((~sure).sum())


def sample_rows(B, n, window, ids, count=4096, seed=0):
    """Seeded query rows for the large workloads: always 0, n-1, window-1 and
    window of every batch, plus members of the largest and smallest groups,
    the rest uniform."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(B):
        for i in (0, n - 1, window - 1, window, n // 2):
            if 0 <= i < n:
                rows.add(b * n + i)
    first = ids[..., 0].reshape(-1)
    sizes = np.bincount(first, minlength=int(first.max()) + 1)
    nonempty = np.nonzero(sizes)[0]
    for g in (int(np.argmax(sizes)), int(nonempty[np.argmin(sizes[nonempty])])):
        members = np.nonzero(first == g)[0]
        pick = rng.choice(members, size=min(64, members.size), replace=False)
        rows.update(int(x) for x in pick)
        rows.add(int(members[-1]))
    while len(rows) < count:
        rows.add(int(rng.integers(0, B * n)))
    return np.array(sorted(rows), dtype=np.int64)


def free_cuda():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
