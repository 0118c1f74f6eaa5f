"""The allocation-free step, for callers that must not allocate GPU memory.

Some callers cannot create a context, because adamw_create allocates: code
that runs inside a framework or server owning all device memory through its
own pool, plug-ins given only their input and output buffers, and
latency-critical paths where cudaMalloc would synchronise the device.  They
call adamw_clip_step_noalloc, whose scratch is a fixed static device array.

These checks call it through the C ABI and compare it with the context-based
adamw_clip_step on two calls in a row: the same bits for w, m, v and the
norm, as its declaration promises (it runs the same kernels with the same
host scalars).  One case also compares every element with the oracle.  This
file is collected last; it passes alone in a fresh process and after the
other tests (the shared array keeps the last call's contents, and each call
clears what must start at zero)."""
import numpy as np
import pytest

import synthetic
from parity import RTOL_NORM, RTOL_ONE_STEP, assert_state_close

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

LR, WD, CLIP = 3e-3, 0.01, 1.0


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _grad(n, t, dev):
    return torch.from_numpy(synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01,
                                            outlier_mult=100.0)).to(dev)


def _views(dev, n, offset):
    """w, m, v as views starting `offset` floats into larger buffers (offset
    1: 4-byte but not 16-byte aligned, the scalar kernels)."""
    out = []
    for i, x in enumerate((synthetic.weights(7, n=n), np.zeros(n, np.float32),
                           np.zeros(n, np.float32))):
        buf = torch.zeros(n + 4, device=dev)
        buf[offset:offset + n] = torch.from_numpy(x).to(dev)
        out.append(buf[offset:offset + n])
    return out


def _assert_same_bits(a, b, label):
    for name, x, y in zip("wmv", a, b):
        assert torch.equal(x, y), f"{label}: {name} differs"


@pytest.mark.parametrize("n", [65536 + 37, 1_000_003, (1 << 24) + 5])
def test_noalloc_step_equals_context_step_bit_for_bit(dev, n):
    """(2^24 + 5: the context step hands chunks out by its counter, the
    no-alloc step keeps the fixed assignment -- the same bits either way.)"""
    states = [_views(dev, n, 0) for _ in range(2)]
    norm_out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in (1, 2):  # two calls in a row
            g = _grad(n, t, dev)
            w, m, v = states[0]
            osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            ref_norm, _ = osr.adamw_last_norm(ctx)
            w, m, v = states[1]
            osr.adamw_clip_step_noalloc(w, g, m, v, t, LR, WD, CLIP, norm_out=norm_out)
            torch.cuda.synchronize()
            assert float(norm_out.item()) == ref_norm, (t, float(norm_out.item()), ref_norm)
            _assert_same_bits(states[0], states[1], f"n={n} t={t}")


@pytest.mark.parametrize("offset", [1, 3])
def test_noalloc_unaligned_views_take_the_scalar_path(dev, offset):
    """Views 4 bytes (12 bytes) past a 16-byte boundary: the scalar norm load
    and the scalar update kernel, in both paths."""
    n = 100_003
    states = [_views(dev, n, offset) for _ in range(2)]
    gbuf = torch.zeros(n + 4, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in (1, 2):
            gbuf[offset:offset + n] = _grad(n, t, dev)
            g = gbuf[offset:offset + n]
            w, m, v = states[0]
            osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            w, m, v = states[1]
            osr.adamw_clip_step_noalloc(w, g, m, v, t, LR, WD, CLIP)  # no norm_out
            torch.cuda.synchronize()
            _assert_same_bits(states[0], states[1], f"offset={offset} t={t}")


def test_noalloc_hyperparameters_given_per_call(dev):
    """beta1, beta2, eps passed to each call equal a context's
    adamw_set_hparams, bit for bit."""
    n = 300_007
    b1, b2, eps = 0.8, 0.95, 1e-6
    states = [_views(dev, n, 0) for _ in range(2)]
    norm_out = torch.zeros(1, dtype=torch.float64, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_hparams(ctx, b1, b2, eps)
        for t in (1, 2, 3):
            g = _grad(n, t, dev)
            w, m, v = states[0]
            osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            ref_norm, _ = osr.adamw_last_norm(ctx)
            w, m, v = states[1]
            osr.adamw_clip_step_noalloc(w, g, m, v, t, LR, WD, CLIP, beta1=b1, beta2=b2,
                                        eps=eps, norm_out=norm_out)
            torch.cuda.synchronize()
            assert float(norm_out.item()) == ref_norm
            _assert_same_bits(states[0], states[1], f"hparams t={t}")


@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_noalloc_nonfinite_gradient_leaves_the_state(dev, bad):
    """A non-finite gradient: w, m, v keep their bits and the norm written to
    norm_out is not finite; the next call with a finite gradient steps."""
    n = 70_001
    w, m, v = _views(dev, n, 0)
    m.copy_(torch.from_numpy(synthetic.draw(7, 11, 0, 1e-3, n=n)).to(dev))
    v.copy_(torch.from_numpy(np.abs(synthetic.draw(7, 12, 0, 1e-5, n=n))).to(dev))
    before = [x.clone() for x in (w, m, v)]
    g = _grad(n, 1, dev)
    g[n // 3] = bad
    norm_out = torch.zeros(1, dtype=torch.float64, device=dev)
    osr.adamw_clip_step_noalloc(w, g, m, v, 5, LR, WD, CLIP, norm_out=norm_out)
    torch.cuda.synchronize()
    assert not np.isfinite(float(norm_out.item()))
    _assert_same_bits((w, m, v), before, "non-finite gradient")
    g[n // 3] = 0.0
    osr.adamw_clip_step_noalloc(w, g, m, v, 5, LR, WD, CLIP, norm_out=norm_out)
    torch.cuda.synchronize()
    assert np.isfinite(float(norm_out.item()))
    assert not torch.equal(w, before[0])


def test_noalloc_every_element_against_the_oracle(dev, oracle):
    """2^24 + 5 parameters, t = 7, generator-made non-zero moments: every
    element of w, m, v within the one-step bar of the oracle's double
    arithmetic, the norm within 1e-6, on two calls in a row (the second
    from the first call's oracle state, so no GPU value reaches the
    oracle)."""
    n = (1 << 24) + 5
    hw = synthetic.weights(7, n=n)
    hm = synthetic.draw(7, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(7, 12, 0, 1e-5, n=n))
    norm_out = torch.zeros(1, dtype=torch.float64, device=dev)
    ow, om, ov = hw.copy(), hm.copy(), hv.copy()
    w, m, v = (torch.from_numpy(x.copy()).to(dev) for x in (hw, hm, hv))
    idx = np.arange(n)
    for t in (7, 8):
        hg = synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
        g = torch.from_numpy(hg).to(dev)
        osr.adamw_clip_step_noalloc(w, g, m, v, t, LR, WD, CLIP, norm_out=norm_out)
        torch.cuda.synchronize()
        onorm = oracle.global_norm(hg)
        assert abs(float(norm_out.item()) - onorm) <= RTOL_NORM * onorm
        s = oracle.clip_scale(onorm, CLIP)
        terms = oracle.adamw_terms_at(idx, ow, hg, om, ov, s, t, LR, WD)
        want = oracle.adamw_at(idx, ow, hg, om, ov, s, t, LR, WD)
        got = [x.cpu().numpy() for x in (w, m, v)]
        assert_state_close(got, want, terms, RTOL_ONE_STEP, f"noalloc t={t}", lr=LR, t=t)
        del terms
        # both sides continue from their own state; the second call's inputs
        # to the oracle are the oracle's own first-call results
        ow, om, ov = want
        w, m, v = (torch.from_numpy(x.copy()).to(dev) for x in want)


def test_noalloc_rejects_sizes_beyond_its_limit(dev):
    lib = osr.library()
    x = torch.zeros(4, device=dev)
    p = x.data_ptr()
    for n in (0, -5, 1 << 31):
        st = lib.adamw_clip_step_noalloc(p, p, p, p, n, 1, 1e-3, 0.0, 1.0, 0.9, 0.999, 1e-8,
                                         None, torch.cuda.current_stream().cuda_stream)
        assert st == osr.EINVAL
        assert "2^31-1" in osr.adamw_last_error()
