"""Element-wise comparison against the oracle with the tolerance contract
|x - ref| <= atol + rtol |ref| (bf16 outputs and gradients: atol = rtol =
1e-2), lse within 1e-4 max(1, |ref|), exact -inf and exact zeros on empty rows,
every value finite.  Failures report the max and mean error and the first
failing coordinates ("attention-algorithm-error-and-complexity-tests", second
paragraph)."""
import math

import numpy as np

ATOL = 1e-2
RTOL = 1e-2
LSE_TOL = 1e-4


def to_np(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def check_close(name, got, ref, atol=ATOL, rtol=RTOL, stats=None):
    got, ref = to_np(got), to_np(ref)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values at {np.argwhere(~np.isfinite(got))[:5]}"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if stats is not None:
        stats[name] = {"max_abs": float(err.max(initial=0.0)),
                       "mean_abs": float(err.mean()) if err.size else 0.0}
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = ", ".join(f"{tuple(i)}: got {got[tuple(i)]:.6g} ref {ref[tuple(i)]:.6g}" for i in idx)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"max err {err.max():.3g}, mean {err.mean():.3g}; {detail}")


def check_lse(name, got, ref, stats=None):
    got, ref = to_np(got), to_np(ref)
    assert got.shape == ref.shape
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf_ref), \
        f"{name}: -inf pattern differs at {np.argwhere(np.isneginf(got) != ninf_ref)[:5]}"
    fin = ~ninf_ref
    assert np.all(np.isfinite(got[fin])), f"{name}: non-finite lse"
    err = np.abs(got[fin] - ref[fin])
    tol = LSE_TOL * np.maximum(1.0, np.abs(ref[fin]))
    if stats is not None:
        stats[name] = {"max_abs": float(err.max(initial=0.0))}
    if (err > tol).any():
        i = int(np.argmax(err - tol))
        raise AssertionError(f"{name}: lse error {err.max():.3g} (worst got {got[fin][i]} ref {ref[fin][i]})")
