"""Tolerances and helpers of the GPU-vs-oracle parity tests.

Bars (the optimizer step's floating point is float32 on the GPU and double
on the oracle):

* gradient norm: |norm_gpu - norm_oracle| <= 1e-6 * norm_oracle.
* w, m, v after one step: relative to the magnitude of the terms that form
  each value, because the new weight is a difference
  w (1 - lr wd) - update that can cancel to ~0, and the new moment a sum
  beta1 m + (1 - beta1) g_hat that can cancel too.  Per element:
      M     = max(|m'|, beta1 |m|, (1 - beta1) |g_hat|)
      |dm| <= rtol * M
      |dv| <= rtol * |v'|                 (all terms of v are >= 0)
      |dw| <= rtol * max(|w'|, |w (1 - lr wd)|, |update|, U)
      U     = lr / (1 - beta1^t) * M / (sqrt(v_hat) + eps)
  U is the update evaluated at m's largest term: when m' cancels, its
  float32 rounding error (a fraction of M, not of |m'|) reaches the update
  through m_hat, so the weight's error scales with U.
  Each bound also allows 2^-148 absolute (two float32 subnormal units) for
  results that underflow.  rtol = 1e-6 after one step.
* Along a trajectory (rtol = 1e-5 after up to 80 steps), an element's error
  is what earlier steps left in it, multiplied by the factor its value has
  been multiplied by since (beta1 for m, beta2 for v, 1 - lr wd for w), plus
  the new rounding.  So the magnitude is carried the same way
  (``Running``): R_m(t) = max(M(t), beta1 R_m(t-1)), R_v(t) =
  max(|v'(t)|, beta2 R_v(t-1)), R_w(t) = max(W(t), (1 - lr wd) R_w(t-1)),
  with W(t) the one-step weight magnitude whose U uses R_m(t).

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
BETA2 = 0.999
EPS = 1e-8


def magnitudes(terms: np.ndarray, lr: float, t: int, beta1: float = BETA1,
               eps: float = EPS):
    """Per-element term magnitudes of w', m', v' from oracle terms (k, 8)."""
    gh, m, v, _mh, vh, wdec, upd, w = terms.T
    carried = np.abs(m - (1.0 - beta1) * gh)  # = beta1 |m_old|
    mag_m = np.maximum(np.maximum(np.abs(m), carried), (1.0 - beta1) * np.abs(gh))
    upd_at_m_terms = lr / (1.0 - beta1 ** t) * mag_m / (np.sqrt(vh) + eps)
    mag_w = np.maximum.reduce([np.abs(w), np.abs(wdec), np.abs(upd), upd_at_m_terms])
    mag_v = np.abs(v)
    return mag_w, mag_m, mag_v


def assert_state_close(got, want, terms, rtol, label="", *, lr, t, beta1=BETA1, eps=EPS):
    """got/want: (w, m, v) float32 arrays at the same indices; terms: the
    oracle's double terms of the step (update t, learning rate lr) that
    produced want from inputs both sides shared."""
    assert_within(got, want, magnitudes(terms, lr, t, beta1, eps), rtol, label)


class Running:
    """Term magnitudes carried along an oracle trajectory (see above)."""

    def __init__(self, beta1=BETA1, beta2=BETA2, eps=EPS):
        self.beta1, self.beta2, self.eps = beta1, beta2, eps
        self.r = None

    def update(self, terms, lr, wd, t):
        """Folds in the oracle's terms of step t; returns (R_w, R_m, R_v)."""
        gh, m, v, _mh, vh, wdec, upd, w = terms.T
        b1 = self.beta1
        mag_m = np.maximum.reduce([np.abs(m), np.abs(m - (1.0 - b1) * gh),
                                   (1.0 - b1) * np.abs(gh)])
        mag_v = np.abs(v)
        if self.r is not None:
            mag_m = np.maximum(mag_m, b1 * self.r[1])
            mag_v = np.maximum(mag_v, self.beta2 * self.r[2])
        u_at_m = lr / (1.0 - b1 ** t) * mag_m / (np.sqrt(vh) + self.eps)
        mag_w = np.maximum.reduce([np.abs(w), np.abs(wdec), np.abs(upd), u_at_m])
        if self.r is not None:
            mag_w = np.maximum(mag_w, (1.0 - lr * wd) * self.r[0])
        self.r = (mag_w, mag_m, mag_v)
        return self.r


def assert_within(got, want, mags, rtol, label=""):
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


def relative_error_report(got, want, terms, *, lr, t, beta1=BETA1, eps=EPS):
    """max err / term magnitude per array (for logs)."""
    out = {}
    for name, g, o, mag in zip("wmv", got, want, magnitudes(terms, lr, t, beta1, eps)):
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
