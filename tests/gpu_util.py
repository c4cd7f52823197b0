"""Shared helpers of the GPU tests: the tolerances and the comparisons against the oracle."""
from __future__ import annotations

import numpy as np

from paged_fp8_kv_04_gb300.synth import rows_of, subset  # noqa: F401  (re-exported)

# bf16 outputs against the fp64 oracle (max-abs and cosine); LSE in natural-log units.
MAX_ABS = 1e-2
MIN_COS = 0.9999
LSE_ABS = 2e-3
# split-K against single pass, both fp32 outputs: element by element, relative to the
# element, with a floor of the same fraction of the largest element of its (row, head)
# (an element near zero cannot be judged relative to itself: two schedules round each P
# term to f16 independently, a noise of ~2e-4 of the row's RMS per element)
SPLIT_REL = 1e-3


def _per_head(a):
    """[rows, heads, D] -> [rows * heads, D]."""
    a = np.asarray(a, dtype=np.float64)
    return a.reshape(-1, a.shape[-1]) if a.ndim >= 2 else a.reshape(1, -1)


def compare(got, ref, what="", max_abs=MAX_ABS, min_cos=MIN_COS, rel_rows=False):
    """Every output finite; max-abs error <= max_abs (relative to each (row, head)'s
    largest |ref| when rel_rows); cosine >= min_cos for every (row, head) vector (a zero
    reference vector must come back as zeros)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if not got.size:
        return 0.0, 1.0
    g, r = _per_head(got), _per_head(ref)
    diff = np.abs(g - r)
    if rel_rows:
        scale = np.abs(r).max(axis=1)
        zero = scale == 0
        assert np.all(diff[zero] == 0), f"{what}: nonzero output where the oracle's is zero"
        rel = diff[~zero].max(axis=1) / scale[~zero]
        err = float(rel.max()) if rel.size else 0.0
        worst = int(np.flatnonzero(~zero)[np.argmax(rel)]) if rel.size else -1
        assert err <= max_abs, f"{what}: (row, head) {divmod(worst, got.shape[1])}: rel err {err:.3e} > {max_abs}"
    else:
        err = float(diff.max())
        assert err <= max_abs, f"{what}: max abs {err:.3e} > {max_abs} at {np.unravel_index(np.argmax(np.abs(got - ref)), got.shape)}"
    ng, nr = np.linalg.norm(g, axis=1), np.linalg.norm(r, axis=1)
    both = (ng > 0) & (nr > 0)
    assert np.array_equal(ng > 0, nr > 0), f"{what}: a (row, head) is zero on one side only"
    cos = (g[both] * r[both]).sum(axis=1) / (ng[both] * nr[both])
    cmin = float(cos.min()) if cos.size else 1.0
    if cos.size:
        worst = int(np.flatnonzero(both)[np.argmin(cos)])
        assert cmin >= min_cos, f"{what}: (row, head) {divmod(worst, got.shape[1])}: cosine {cmin:.7f} < {min_cos}"
    return err, cmin


def compare_split(a, b, what="", rel=SPLIT_REL):
    """fp32 outputs of two schedules, element by element: |a - b| <= rel * (|b| + the
    largest |b| of the element's (row, head) vector)."""
    a, b = _per_head(a), _per_head(b)
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b)), f"{what}: non-finite output"
    rowmax = np.abs(b).max(axis=1, keepdims=True)
    bound = rel * (np.abs(b) + rowmax)
    bad = np.abs(a - b) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond {rel} relative; worst "
                           f"{float((np.abs(a - b) / np.maximum(bound / rel, 1e-300)).max()):.3e}")


def compare_lse(got, ref, what="", tol=LSE_ABS, rel=0.0):
    """|got - ref| <= tol + rel * |ref| for every finite lse, and the same infinities."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: lse finiteness differs"
    if fin.any():
        excess = np.abs(got[fin] - ref[fin]) - (tol + rel * np.abs(ref[fin]))
        assert excess.max() <= 0, f"{what}: lse err beyond its bound by {float(excess.max()):.3e}"
