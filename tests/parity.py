"""Tolerances for comparing the CUDA path with the fp64 oracle.

fp32 results: |g - o| <= 1e-6 + 1e-5 * max(|o|, c / sqrt(n)), where c is the
oracle's conditioning scale of the output (sum of |terms|) and n the number
of terms; with c unavailable this is the plain allclose(rtol=1e-5, atol=1e-6).
The c/sqrt(n) floor only matters for outputs that are a cancelling sum of
O(1) terms, where fp32 accumulation alone cannot reach 1e-5 of |o|.

bf16 results (fp32 accumulation, bf16 rounding of the output):
|g - o| <= 1e-2 * |o| + 1e-4 * c. The relative part covers the bf16 rounding
(2^-9); the absolute part covers fp32 accumulation and score rounding near
o = 0 with a 10x margin over the worst-case bound of a 4096-term row.

Both return the fraction that meets the strict relative form (no c term), so
tests can report it alongside.
"""
import json
import os

import numpy as np


def _log(name, strict, n):
    """Append the strict-allclose pass fraction of one comparison to the JSON
    lines file named by GAT_PARITY_LOG (nothing when it is unset), so a run
    records how far each case is from the plain rtol/atol criterion."""
    path = os.environ.get("GAT_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, "strict_fraction": strict, "n": int(n)}) + "\n")


def _report(name, g, o, tol):
    err = np.abs(g - o)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        lines = [f"  at {tuple(i)}: got {g[tuple(i)]!r} want {o[tuple(i)]!r} tol {tol[tuple(i)]!r}"
                 for i in idx]
        raise AssertionError(f"{name}: {int(bad.sum())} of {g.size} outside tolerance, "
                             f"max err {np.nanmax(err):.3e}\n" + "\n".join(lines))


def assert_fp32(g, o, cond=None, n_terms=None, name="fp32"):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    scale = np.abs(o)
    if cond is not None:
        n = np.maximum(np.asarray(n_terms if n_terms is not None else 1, dtype=np.float64), 1.0)
        scale = np.maximum(scale, np.asarray(cond) / np.sqrt(n))
    nan_o = np.isnan(o)
    tol = np.where(nan_o, np.inf, 1e-6 + 1e-5 * scale)
    assert (np.isnan(g) == nan_o).all(), f"{name}: NaN pattern differs"
    _report(name, np.where(nan_o, 0, g), np.where(nan_o, 0, o), tol)
    strict = np.abs(g - o) <= 1e-6 + 1e-5 * np.abs(o)
    rate = float(np.mean(strict[~nan_o])) if (~nan_o).any() else 1.0
    _log(name, rate, (~nan_o).sum())
    return rate


def assert_bf16(g, o, cond, name="bf16"):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    tol = 1e-2 * np.abs(o) + 1e-4 * np.asarray(cond)
    _report(name, g, o, tol)
    strict = np.abs(g - o) <= 1e-2 * np.abs(o)
    rate = float(np.mean(strict))
    _log(name, rate, g.size)
    return rate
