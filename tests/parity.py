"""Tolerances and helpers of the GPU-vs-oracle parity tests.

Bars (the optimizer step's floating point is float32 on the GPU and double
on the oracle):

* gradient norm: |norm_gpu - norm_oracle| <= 1e-6 * norm_oracle.
* w, m, v after one step: relative to the magnitude of the terms that form
  each value, because the new weight is a difference
  w (1 - lr wd) - update that can cancel to ~0, and the new moment a sum
  beta1 m + (1 - beta1) g_hat that can cancel too.  Per element:
      |dw| <= rtol * max(|w'|, |w (1 - lr wd)|, |update|)
      |dm| <= rtol * max(|m'|, beta1 |m|, (1 - beta1) |g_hat|)
      |dv| <= rtol * |v'|                 (all terms of v are >= 0)
  plus 2^-148 absolute (two float32 subnormal units) for results that
  underflow.  rtol = 1e-6 after one step, 1e-5 after 80 steps (term
  magnitudes from the oracle's own last step).

Derivation of the 1e-6 bar: the fused kernel rounds about eight times along
the longest chain (g_hat, the second moment, square root, its scaling plus
eps, division, step size, decay fma), each at most 2^-24 relative, i.e.
about 4.8e-7 of the largest term, plus the norm's own <= 3.6e-7 through the
clip factor for m and v; the oracle's final rounding to float32 adds 6e-8.
"""
from __future__ import annotations

import numpy as np

RTOL_ONE_STEP = 1e-6
RTOL_TRAJECTORY = 1e-5
RTOL_NORM = 1e-6
FLOOR = 2.0 ** -148
BETA1 = 0.9


def magnitudes(terms: np.ndarray, beta1: float = BETA1):
    """Per-element term magnitudes of w', m', v' from oracle terms (k, 8)."""
    gh, m, v, _mh, _vh, wdec, upd, w = terms.T
    mag_w = np.maximum(np.maximum(np.abs(w), np.abs(wdec)), np.abs(upd))
    carried = np.abs(m - (1.0 - beta1) * gh)  # = beta1 |m_old|
    mag_m = np.maximum(np.maximum(np.abs(m), carried), (1.0 - beta1) * np.abs(gh))
    mag_v = np.abs(v)
    return mag_w, mag_m, mag_v


def assert_state_close(got, want, terms, rtol, label=""):
    """got/want: (w, m, v) float32 arrays at the same indices; terms: the
    oracle's double terms of the step that produced want."""
    mags = magnitudes(terms)
    for name, g, o, mag in zip("wmv", got, want, mags):
        err = np.abs(np.asarray(g, np.float64) - np.asarray(o, np.float64))
        bound = rtol * mag + FLOOR
        bad = np.nonzero(~(err <= bound))[0]
        if bad.size:
            i = bad[np.argmax(err[bad] / np.maximum(bound[bad], 1e-300))]
            raise AssertionError(
                f"{label} {name}: {bad.size} of {err.size} elements beyond "
                f"rtol={rtol:g} x term magnitude; worst at {i}: got {g[i]!r} "
                f"want {o[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")


def relative_error_report(got, want, terms):
    """max err / term magnitude per array (for logs)."""
    out = {}
    for name, g, o, mag in zip("wmv", got, want, magnitudes(terms)):
        err = np.abs(np.asarray(g, np.float64) - np.asarray(o, np.float64))
        out[name] = float(np.max(err / np.maximum(mag, 1e-300)))
    return out


def sample_indices(n: int, k: int, seed: int = 0) -> np.ndarray:
    """Sorted distinct indices: the first and last few, tile edges, random."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 2, 3, 4, 5, n - 1, n - 2, n - 3, n - 4, n // 2]
    for b in (8192, 1 << 20):
        for e in range(b, n, max(b, n // 64)):
            fixed += [e - 1, e]
    idx = np.concatenate([np.array([i for i in fixed if 0 <= i < n], np.int64),
                          rng.integers(0, n, size=min(k, n), dtype=np.int64)])
    return np.unique(idx)
