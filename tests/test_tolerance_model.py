"""The parity bounds of ``parity.py`` hold for the fused kernel's float32
operation sequence, emulated here in numpy (each float32 op correctly
rounded; fused multiply-adds as an exact double product plus one rounding),
on random states and on states built to cancel.  This checks the tolerance
derivation on the CPU; the GPU tests check the kernel itself."""
import numpy as np
import pytest

from parity import RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, assert_state_close, assert_within

f32 = np.float32


def fma(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(f32)


def kernel_step(w, g, m, v, s, t, lr, wd, b1, b2, eps):
    """The fused kernel's sequence: g_hat, m fma, v fma, denom fma, div,
    step-size multiply, decay fma (scalars rounded to float32 once)."""
    bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
    k_b1, k_omb1, k_b2, k_omb2 = f32(b1), f32(1 - b1), f32(b2), f32(1 - b2)
    k_eps, k_step, k_isb, k_dec = f32(eps), f32(lr / bc1), f32(1 / np.sqrt(bc2)), f32(1 - lr * wd)
    gh = (g * f32(s)).astype(f32)
    m2 = fma(np.full_like(m, k_b1), m, (k_omb1 * gh).astype(f32))
    v2 = fma(np.full_like(v, k_b2), v, ((k_omb2 * gh).astype(f32) * gh).astype(f32))
    den = fma(np.sqrt(v2).astype(f32), np.full_like(v2, k_isb), np.full_like(v2, k_eps))
    upd = (k_step * (m2 / den).astype(f32)).astype(f32)
    w2 = fma(w, np.full_like(w, k_dec), -upd)
    return w2, m2, v2


@pytest.mark.parametrize("case", ["random", "m_cancels", "w_cancels", "tiny_v", "hparams"])
def test_bound_holds_for_kernel_arithmetic(oracle, case):
    rng = np.random.default_rng(hash(case) % 2**32)
    n = 200_000
    b1, b2, eps, lr, wd, t = 0.9, 0.999, 1e-8, 3e-3, 0.01, 7
    w = rng.normal(0, 0.02, n).astype(f32)
    g = rng.normal(0, 1e-2, n).astype(f32)
    m = rng.normal(0, 1e-3, n).astype(f32)
    v = np.abs(rng.normal(0, 1e-5, n)).astype(f32)
    if case == "m_cancels":      # beta1 m ~ -(1 - beta1) g_hat
        m = (-(1 - b1) / b1 * g * rng.uniform(0.999, 1.001, n)).astype(f32)
    elif case == "w_cancels":    # w (1 - lr wd) ~ update
        w = (lr * np.sign(g) * rng.uniform(0.5, 2.0, n)).astype(f32)
    elif case == "tiny_v":
        v = np.abs(rng.normal(0, 1e-30, n)).astype(f32)
        g = (g * 1e-6).astype(f32)
    elif case == "hparams":
        b1, b2, eps, lr, wd, t = 0.5, 0.75, 1e-6, 1e-2, 0.1, 3
        m = (-(1 - b1) / b1 * g * rng.uniform(0.99, 1.01, n)).astype(f32)
    s = oracle.clip_scale(oracle.global_norm(g), 1.0)
    got = kernel_step(w, g, m, v, s, t, lr, wd, b1, b2, eps)
    idx = np.arange(n)
    want = oracle.adamw_at(idx, w, g, m, v, s, t, lr, wd, b1, b2, eps)
    terms = oracle.adamw_terms_at(idx, w, g, m, v, s, t, lr, wd, b1, b2, eps)
    assert_state_close(got, want, terms, RTOL_ONE_STEP, case, lr=lr, t=t, beta1=b1, eps=eps)


@pytest.mark.parametrize("outliers", [True, False])
def test_trajectory_bound_holds_for_kernel_arithmetic(oracle, outliers):
    """80 steps of the flat-65536 workload: the emulated kernel state stays
    within the carried-magnitude bound of the oracle's trajectory at every
    step; the clip factor is perturbed by the norm's worst-case error
    (3.6e-7 for the float32 runs of the sum of squares, halved by the root)."""
    import synthetic
    from synthetic import workloads as W
    wl = W.flat_65k()
    n = wl.n
    w = synthetic.weights(wl.seed, n=n)
    m = np.zeros(n, f32)
    v = np.zeros(n, f32)
    ow, om, ov = w.copy(), m.copy(), v.copy()
    run = Running()
    idx = np.arange(n)
    for t in range(1, wl.steps + 1):
        g = synthetic.grads(wl.seed, t, wl.grad_sigma, n=n,
                            outlier_frac=wl.outlier_frac if outliers else 0.0,
                            outlier_mult=wl.outlier_mult)
        s = oracle.clip_scale(oracle.global_norm(g), wl.clip)
        w, m, v = kernel_step(w, g, m, v, s * (1 + 1.8e-7), t, wl.lr, wl.wd, 0.9, 0.999, 1e-8)
        mags = run.update(oracle.adamw_terms_at(idx, ow, g, om, ov, s, t, wl.lr, wl.wd),
                          wl.lr, wl.wd, t)
        oracle.adamw_clip_step(ow, g, om, ov, t, wl.lr, wl.wd, wl.clip)
        rtol = RTOL_ONE_STEP if t == 1 else RTOL_TRAJECTORY
        assert_within((w, m, v), (ow, om, ov), mags, rtol, f"step {t}")
