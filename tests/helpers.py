"""Comparison helpers shared by the GPU parity tests.

float32 inputs: max over elements of |got - want| / max(|want|, 1e-3 max|want|)
must stay below 1e-4.

bfloat16 inputs (float32 accumulation): phi(q), phi(k) and the intra-chunk
weights enter the tensor cores rounded to bf16, which perturbs every weight by
~2^-9 relative. Outputs are convex combinations of v (and gradients sums of
such terms), so that perturbation is an absolute error on the scale of the
largest terms, not of each output element; an element that happens to sit
near zero cannot keep a small relative error in any bf16 computation. The
2e-2 bound is therefore applied (a) normwise, max|got - want| / max|want|,
and (b) elementwise on the significant elements, |want| >= 0.1 max|want|.
"""

import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}
SIGNIFICANT = 0.1


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def max_rel_err(got, want, floor=1e-3):
    """max_e |got - want| / max(|want|, floor * max|want|)."""
    got, want = _f64(got), _f64(want)
    assert got.shape == want.shape, (got.shape, want.shape)
    if want.size == 0:
        return 0.0
    fl = floor * max(float(np.max(np.abs(want))), 1e-300)
    return float(np.max(np.abs(got - want) / np.maximum(np.abs(want), fl)))


def normwise_err(got, want):
    got, want = _f64(got), _f64(want)
    if want.size == 0:
        return 0.0
    return float(np.max(np.abs(got - want)) / max(float(np.max(np.abs(want))), 1e-300))


def significant_rel_err(got, want, frac=SIGNIFICANT):
    got, want = _f64(got), _f64(want)
    if want.size == 0:
        return 0.0
    sel = np.abs(want) >= frac * np.max(np.abs(want))
    return float(np.max(np.abs(got[sel] - want[sel]) / np.abs(want[sel])))


def errors(got, want, dtype):
    if dtype == "f32":
        return {"max_rel": max_rel_err(got, want)}
    return {"normwise": normwise_err(got, want), "significant_rel": significant_rel_err(got, want)}


# Every comparison's errors, by dtype: the session summary (conftest.py) prints the
# largest of each, with the plain elementwise relative error of the bf16 cases
# (not a pass criterion, so that its gap to the criteria above stays visible).
RECORD = {"f32": {}, "bf16": {}}


def _record(dtype, errs, what):
    book = RECORD[dtype]
    for key, val in errs.items():
        if key not in book or val > book[key][0]:
            book[key] = (val, what)


def assert_close(got, want, dtype, what=""):
    if np.any(~np.isfinite(_f64(got))):
        raise AssertionError(f"{what}: non-finite values")
    errs = errors(got, want, dtype)
    report = dict(errs)
    if dtype == "bf16":
        report["plain_max_rel (reported only)"] = max_rel_err(got, want)
    _record(dtype, report, what)
    bad = {k: v for k, v in errs.items() if not v < TOL[dtype]}
    assert not bad, f"{what}: {report} (tolerance {TOL[dtype]})"
    return errs
