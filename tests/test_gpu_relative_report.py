"""Transparency report on the parity bar: how many elements would fail a
pure relative test (|got - want| <= rtol |want|) although they meet the
term-magnitude bar the parity tests use (tests/parity.py).  Every such
element must be one whose value is smaller than the terms that form it (a
cancellation), which is what the term-magnitude bar exists for.  The counts
are printed (pytest -s).  Along the flat-65536 trajectory they grow with t:
weights move about lr = 3e-3 per step around values of about 0.02, so many
cross zero, where w (1 - lr wd) and the update cancel."""
import numpy as np
import pytest

import synthetic
from synthetic import workloads as W
from parity import FLOOR, RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, assert_within

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def pure_relative_failures(got, want, mags, rtol):
    """Per array: indices failing |d| <= rtol |want| (want != 0), checked to
    be cancellations (|want| below the term magnitude)."""
    out = {}
    for name, g, o, mag in zip("wmv", got, want, mags):
        g = np.asarray(g, np.float64)
        o = np.asarray(o, np.float64)
        err = np.abs(g - o)
        bad = np.nonzero(err > rtol * np.abs(o))[0]
        bad = bad[o[bad] != 0.0] if bad.size else bad
        # the term bar allows err <= rtol mag + FLOOR, so failing the pure
        # test means |want| < mag + FLOOR / rtol
        assert np.all(np.abs(o[bad]) < mag[bad] + FLOOR / rtol), name
        out[name] = int(bad.size)
    return out


def test_flat_65536_trajectory_counts(dev, oracle):
    wl = W.flat_65k()
    n = wl.n
    hw = synthetic.weights(wl.seed, n=n)
    ow, om, ov = hw.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    w = torch.from_numpy(hw).to(dev)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    idx = np.arange(n)
    run = Running()
    report = {}
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in range(1, wl.steps + 1):
            gh = synthetic.grads(wl.seed, t, wl.grad_sigma, n=n, outlier_frac=wl.outlier_frac,
                                 outlier_mult=wl.outlier_mult)
            osr.adamw_clip_step(ctx, w, torch.from_numpy(gh).to(dev), m, v, t, wl.lr, wl.wd,
                                wl.clip)
            s = oracle.clip_scale(oracle.global_norm(gh), wl.clip)
            terms = oracle.adamw_terms_at(idx, ow, gh, om, ov, s, t, wl.lr, wl.wd)
            mags = run.update(terms, wl.lr, wl.wd, t)
            oracle.adamw_clip_step(ow, gh, om, ov, t, wl.lr, wl.wd, wl.clip)
            if t in (1, 10, 40, 80):
                got = [x.cpu().numpy() for x in (w, m, v)]
                rtol = RTOL_ONE_STEP if t == 1 else RTOL_TRAJECTORY
                assert_within(got, (ow, om, ov), mags, rtol, f"t={t}")
                report[t] = pure_relative_failures(got, (ow, om, ov), mags, rtol)
    print(f"\nflat-65536, elements failing a pure relative test (of {n}): {report}")
    assert all(c["v"] == 0 for c in report.values())  # v has no cancelling terms


def test_one_step_counts_nonzero_moments(dev, oracle):
    """One step from generator states with non-zero moments (where m can
    cancel), 1,000,003 elements."""
    n = 1_000_003
    hw = synthetic.weights(7, n=n)
    hm = synthetic.draw(7, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(7, 12, 0, 1e-5, n=n))
    hg = synthetic.grads(7, 3, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
    t, lr, wd = 5, 3e-3, 0.01
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step(ctx, w, g, m, v, t, lr, wd, 1.0)
    s = oracle.clip_scale(oracle.global_norm(hg), 1.0)
    idx = np.arange(n)
    want = oracle.adamw_at(idx, hw, hg, hm, hv, s, t, lr, wd)
    terms = oracle.adamw_terms_at(idx, hw, hg, hm, hv, s, t, lr, wd)
    mags = Running().update(terms, lr, wd, t)
    got = [x.cpu().numpy() for x in (w, m, v)]
    assert_within(got, want, mags, RTOL_ONE_STEP, "one step")
    counts = pure_relative_failures(got, want, mags, RTOL_ONE_STEP)
    print(f"\n1,000,003 elements, t=5 from non-zero moments, failing a pure relative "
          f"1e-6 test: {counts}")
    assert counts["v"] == 0
