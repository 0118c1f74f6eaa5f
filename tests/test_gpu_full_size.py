"""Every element of one full-size step against the oracle.

The 110M tensor list (196 tensors, n = 110,418,432; the fused kernel hands
its chunks out by a counter at this size) and the flat 2^30-parameter (1B)
state, one step at t = 7 from generator-made non-zero moments, so that both
bias corrections and both moment terms are in play; and the flat 12.8M
configuration's whole 100-step trajectory.  On the 110M list:

* float32 gradient, decay on every parameter;
* decay flags exempting every 1-D tensor (biases, LayerNorm gains and
  shifts): the oracle's per-element definition with wd = 0 on those tensors;
* bfloat16 gradient (widened exactly on both sides) with a bfloat16 copy of
  the new weights, which must be the nearest-even rounding of the GPU's own
  float32 weights.

The oracle evaluates its per-element definition ("Training as a Recoverable
State Transition", section "The Exact Targets of Clipping and AdamW") over
index chunks on all host cores; its clip factor comes from its own norm of
the whole gradient.  Bars: the norm within 1e-6 relative, w, m, v within
1e-6 of their term magnitudes (tests/parity.py)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from synthetic import workloads as W
from parity import FLOOR, RTOL_NORM, RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, magnitudes

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

T = 7
CHUNK = 1 << 21


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _state(dev, n, outlier_frac=0.0, outlier_mult=1.0):
    """w, g (step T), m, v on the device from the input generator."""
    w = torch.empty(n, device=dev)
    g = torch.empty(n, device=dev)
    m = torch.empty(n, device=dev)
    v = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, 7)
    synth_dev.fill_grads(g, 7, T, 1e-3, outlier_frac, outlier_mult)
    synth_dev.fill(m, 7, 11, 0, 1e-3)
    synth_dev.fill(v, 7, 12, 0, 1e-5)
    v.abs_()
    return w, g, m, v


def _chunks(offsets, numels, wd, flags=None):
    """(lo, hi, wd of the range) over the table, no range longer than CHUNK."""
    out = []
    for k, (off, num) in enumerate(zip(offsets, numels)):
        wk = wd if flags is None or flags[k] else 0.0
        for lo in range(off, off + num, CHUNK):
            out.append((lo, min(lo + CHUNK, off + num), wk))
    return out


def _check_all(oracle, got, hw, hg, hm, hv, s, lr, chunks, label):
    """Every element of got = (w, m, v) against the oracle's step."""

    def one(c):
        lo, hi, wk = c
        idx = np.arange(lo, hi, dtype=np.int64)
        terms = oracle.adamw_terms_at(idx, hw, hg, hm, hv, s, T, lr, wk)
        want = oracle.adamw_at(idx, hw, hg, hm, hv, s, T, lr, wk)
        bad = []
        for name, a, o, mag in zip("wmv", got, want, magnitudes(terms, lr, T)):
            err = np.abs(a[lo:hi].astype(np.float64) - o.astype(np.float64))
            over = np.nonzero(~(err <= RTOL_ONE_STEP * mag + FLOOR))[0]
            if over.size:
                i = over[np.argmax(err[over] / (RTOL_ONE_STEP * mag[over] + FLOOR))]
                bad.append(f"{name}: {over.size} elements, worst {lo + i}: got {a[lo + i]!r} "
                           f"want {o[i]!r} magnitude {mag[i]:.3e}")
        return bad

    with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        bad = [b for r in ex.map(one, chunks) for b in r]
    assert not bad, f"{label}: " + "; ".join(bad[:6])


def _run(dev, oracle, mode):
    wl = W.gpt_110m()
    n = wl.n
    off, num = wl.table()
    w, g, m, v = _state(dev, n)
    hw, hg, hm, hv = (x.cpu().numpy() for x in (w, g, m, v))
    flags = W.decay_flags_matrices_only(wl.tensors) if mode == "decay_flags" else None
    w_lp = None
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        if flags is not None:
            osr.adamw_set_decay_mask(ctx, flags)
        if mode == "bf16":
            bits = synthetic.to_bf16_bits(hg)
            hg = (bits.astype(np.uint32) << 16).view(np.float32)  # exact widening
            g16 = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
            w_lp = torch.empty(n, dtype=torch.bfloat16, device=dev)
            osr.adamw_clip_step_mixed(ctx, w, g16, m, v, T, wl.lr, wl.wd, wl.clip, w_lp=w_lp)
        else:
            osr.adamw_clip_step(ctx, w, g, m, v, T, wl.lr, wl.wd, wl.clip)
        norm, _ = osr.adamw_last_norm(ctx)
    onorm = oracle.global_norm(hg)
    assert abs(norm - onorm) <= RTOL_NORM * onorm, (norm, onorm)
    s = oracle.clip_scale(onorm, wl.clip)
    assert s < 1.0  # the clip is active on this workload
    got = [x.cpu().numpy() for x in (w, m, v)]
    _check_all(oracle, got, hw, hg, hm, hv, s, wl.lr, _chunks(off, num, wl.wd, flags),
               f"110M list, {mode}")
    if w_lp is not None:
        lp = w_lp.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(lp, synthetic.to_bf16_bits(got[0]))


@pytest.mark.parametrize("mode", ["f32", "decay_flags", "bf16"])
def test_gpt_110m_one_step_every_element(dev, oracle, mode):
    _run(dev, oracle, mode)
    torch.cuda.empty_cache()


def _host_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def test_flat_1b_one_step_every_element(dev, oracle):
    """The 1B configuration (flat 2^30, g ~ 1e-3 with 0.1% outliers x1000):
    all 1,073,741,824 elements of w, m and v against the oracle."""
    wl = W.flat_pow2(30)
    n = wl.n
    if _host_available_bytes() < (48 << 30):
        pytest.skip("needs about 40 GB of host memory for the host copies and the oracle")
    w, g, m, v = _state(dev, n, wl.outlier_frac, wl.outlier_mult)
    hw, hg, hm, hv = (x.cpu().numpy() for x in (w, g, m, v))
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step(ctx, w, g, m, v, T, wl.lr, wl.wd, wl.clip)
        norm, _ = osr.adamw_last_norm(ctx)
    onorm = oracle.global_norm(hg)
    assert abs(norm - onorm) <= RTOL_NORM * onorm, (norm, onorm)
    s = oracle.clip_scale(onorm, wl.clip)
    assert s < 1.0
    got = [x.cpu().numpy() for x in (w, m, v)]
    del w, g, m, v
    torch.cuda.empty_cache()
    _check_all(oracle, got, hw, hg, hm, hv, s, wl.lr, _chunks([0], [n], wl.wd), "flat 2^30")


def test_flat_12m8_100_step_trajectory_every_element(dev, oracle):
    """The 12.8M configuration (flat, g ~ 1e-3, every step clipped): 100
    steps on the GPU and, beside them, the oracle's own 100-step trajectory
    of every element from the same generator inputs (its clip factor from its
    own norm each step), run in index chunks on all host cores.  Each step's
    norm within 1e-6 of the oracle's; after 100 steps every element of w, m
    and v within the trajectory bar (1e-5 of the magnitudes carried along the
    oracle's trajectory, tests/parity.py)."""
    wl = W.flat_12m8()
    n = wl.n
    w = torch.empty(n, device=dev)
    g = torch.empty(n, device=dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    ow = w.cpu().numpy()
    om = np.zeros(n, np.float32)
    ov = np.zeros(n, np.float32)
    chunk = 1 << 20
    spans = [(lo, min(lo + chunk, n)) for lo in range(0, n, chunk)]
    runs = [Running() for _ in spans]
    mags = [None] * len(spans)

    def advance(i, hg, s, t):
        lo, hi = spans[i]
        idx = np.arange(lo, hi, dtype=np.int64)
        terms = oracle.adamw_terms_at(idx, ow, hg, om, ov, s, t, wl.lr, wl.wd)
        mags[i] = runs[i].update(terms, wl.lr, wl.wd, t)
        nw, nm, nv = oracle.adamw_at(idx, ow, hg, om, ov, s, t, wl.lr, wl.wd)
        ow[lo:hi], om[lo:hi], ov[lo:hi] = nw, nm, nv

    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx, \
            ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        for t in range(1, wl.steps + 1):
            synth_dev.fill_grads(g, wl.seed, t, wl.grad_sigma)
            hg = g.cpu().numpy()
            osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
            onorm = oracle.global_norm(hg)
            s = oracle.clip_scale(onorm, wl.clip)
            list(ex.map(lambda i: advance(i, hg, s, t), range(len(spans))))
            norm, _ = osr.adamw_last_norm(ctx)
            assert abs(norm - onorm) <= RTOL_NORM * onorm, (t, norm, onorm)
    got = [x.cpu().numpy() for x in (w, m, v)]
    full = [np.concatenate([mg[k] for mg in mags]) for k in range(3)]
    for name, a, o, mag in zip("wmv", got, (ow, om, ov), full):
        err = np.abs(a.astype(np.float64) - o.astype(np.float64))
        bad = np.nonzero(~(err <= RTOL_TRAJECTORY * mag + FLOOR))[0]
        assert bad.size == 0, (name, bad.size, int(bad[0]), a[bad[0]], o[bad[0]], mag[bad[0]])
