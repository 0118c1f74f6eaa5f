"""GPU parity of the fused clip+AdamW step against the oracle: one step at
every element for small and ragged sizes, 80-step trajectories, sampled
elements at the full 12.8M / 110M / 2^30 sizes, the non-finite skip, and the
flat-vs-tensor-table invariant.  All calls go through the C ABI."""
import os
import struct

import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from synthetic import workloads as W
from parity import (RTOL_NORM, RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, assert_state_close,
                    assert_within, sample_indices)

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


HOST_GEN_MAX = 1 << 22  # below this, inputs are drawn on the host and uploaded


def draw(dev, n, seed, stream, step, sigma, frac=0.0, mult=1.0):
    """One generator draw as (device tensor, host array), identical bytes.
    Small draws come from the numpy generator (uploaded); large ones from its
    device twin (downloaded), which test_generator_device_twin_is_bit_exact
    shows to be the same function."""
    if n <= HOST_GEN_MAX:
        h = synthetic.draw(seed, stream, step, sigma, n=n, outlier_frac=frac,
                           outlier_mult=mult)
        return torch.from_numpy(h).to(dev), h
    t = torch.empty(n, device=dev)
    synth_dev.fill(t, seed, stream, step, sigma, frac, mult)
    return t, t.cpu().numpy()


def make_state(dev, n, seed=7, m_sigma=0.0, v_sigma=0.0):
    """Initial (w, m, v) from the generator, on device and host."""
    w, hw = draw(dev, n, seed, synthetic.STREAM_W, 0, 0.02)
    if m_sigma:
        m, hm = draw(dev, n, seed, 11, 0, m_sigma)
    else:
        m, hm = torch.zeros(n, device=dev), np.zeros(n, np.float32)
    if v_sigma:
        v, hv = draw(dev, n, seed, 12, 0, v_sigma)
        v.abs_()
        hv = np.abs(hv)
    else:
        v, hv = torch.zeros(n, device=dev), np.zeros(n, np.float32)
    return (w, m, v), (hw, hm, hv)


def grads(dev, n, wl, t, outliers=True):
    if outliers:
        return draw(dev, n, wl.seed, synthetic.STREAM_G, t, wl.grad_sigma,
                    wl.outlier_frac, wl.outlier_mult)
    return draw(dev, n, wl.seed, synthetic.STREAM_G, t, wl.grad_sigma)


def host(*ts):
    return [t.detach().cpu().numpy().copy() for t in ts]


def one_step_check(oracle, ctx, dstate, hstate, g, hg, t, lr, wd, clip):
    """One GPU step from generator inputs, every element vs the oracle."""
    w, m, v = dstate
    w0, m0, v0 = hstate
    osr.adamw_clip_step(ctx, w, g, m, v, t, lr, wd, clip)
    norm, scale = osr.adamw_last_norm(ctx)
    onorm = oracle.global_norm(hg)
    assert abs(norm - onorm) <= RTOL_NORM * onorm
    s = oracle.clip_scale(onorm, clip)
    idx = np.arange(w0.size)
    want = oracle.adamw_at(idx, w0, hg, m0, v0, s, t, lr, wd)
    terms = oracle.adamw_terms_at(idx, w0, hg, m0, v0, s, t, lr, wd)
    assert_state_close(host(w, m, v), want, terms, RTOL_ONE_STEP, f"t={t}", lr=lr, t=t)
    return norm, scale


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 513, 2048, 2049, 65536, 65536 + 37,
                               1_000_003])
def test_one_step_all_elements(dev, oracle, n):
    """One step at t = 1, 2 and 17, each from the generator's (w, m, v)."""
    wl = W.flat_65k()
    g, hg = grads(dev, n, wl, 1)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in (1, 2, 17):
            dstate, hstate = make_state(dev, n, m_sigma=1e-3, v_sigma=1e-5)
            one_step_check(oracle, ctx, dstate, hstate, g, hg, t, wl.lr, wl.wd, wl.clip)


def test_one_step_unaligned_views(dev, oracle):
    """State arrays that are not 16-byte aligned take the scalar kernel."""
    n = 40_001
    wl = W.flat_65k()
    hg = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    for t in (1, 2):
        (w0, m0, v0), hstate = make_state(dev, n, m_sigma=1e-3, v_sigma=1e-5)
        bufs = [torch.empty(n + 1, device=dev) for _ in range(4)]
        w, g, m, v = (b[1:] for b in bufs)
        assert all(x.data_ptr() % 16 == 4 for x in (w, g, m, v))
        w.copy_(w0)
        m.copy_(m0)
        v.copy_(v0)
        g.copy_(torch.from_numpy(hg))
        with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
            one_step_check(oracle, ctx, (w, m, v), hstate, g, hg, t, wl.lr, wl.wd, wl.clip)


@pytest.mark.parametrize("clip", [float("inf"), 1e6, 1.0, 1e-3])
def test_clip_regimes(dev, oracle, clip):
    n = 70_000
    dstate, hstate = make_state(dev, n)
    g, hg = draw(dev, n, 7, synthetic.STREAM_G, 1, 1e-2)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        norm, scale = one_step_check(oracle, ctx, dstate, hstate, g, hg, 1, 3e-3, 0.01, clip)
        if norm > clip:
            assert abs(scale - clip / norm) <= 1e-7 * (clip / norm)
        else:
            assert scale == 1.0


def test_hparams_and_zero_lr(dev, oracle):
    n = 10_000
    (w, m, v), (w0, m0, v0) = make_state(dev, n, m_sigma=1e-3, v_sigma=1e-5)
    g, g0 = draw(dev, n, 7, synthetic.STREAM_G, 2, 1e-1)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_hparams(ctx, 0.5, 0.75, 1e-6)
        osr.adamw_clip_step(ctx, w, g, m, v, 3, 1e-2, 0.1, 1.0)
        s = oracle.clip_scale(oracle.global_norm(g0), 1.0)
        idx = np.arange(n)
        want = oracle.adamw_at(idx, w0, g0, m0, v0, s, 3, 1e-2, 0.1, 0.5, 0.75, 1e-6)
        terms = oracle.adamw_terms_at(idx, w0, g0, m0, v0, s, 3, 1e-2, 0.1, 0.5, 0.75, 1e-6)
        assert_state_close(host(w, m, v), want, terms, RTOL_ONE_STEP, "hparams",
                           lr=1e-2, t=3, beta1=0.5, eps=1e-6)
        wb = w.clone()
        osr.adamw_clip_step(ctx, w, g, m, v, 4, 0.0, 0.1, 1.0)
        assert torch.equal(w, wb)  # lr = 0 moves nothing (decay is lr * wd)


def test_nonfinite_gradient_skips_the_update(dev):
    n = 30_000
    (w, m, v), _ = make_state(dev, n, m_sigma=1e-3, v_sigma=1e-5)
    g, _ = draw(dev, n, 7, synthetic.STREAM_G, 1, 1e-2)
    g[4321] = float("nan")
    before = [t.clone() for t in (w, m, v)]
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step(ctx, w, g, m, v, 1, 3e-3, 0.01, 1.0)
        with pytest.raises(osr.NonFiniteGradient):
            osr.adamw_last_norm(ctx)
        for a, b in zip((w, m, v), before):
            assert torch.equal(a, b)
        g[4321] = 0.0
        osr.adamw_clip_step(ctx, w, g, m, v, 1, 3e-3, 0.01, 1.0)
        osr.adamw_last_norm(ctx)
        assert not torch.equal(w, before[0])


def test_bad_arguments(dev):
    n = 1000
    (w, m, v), _ = make_state(dev, n)
    g = torch.zeros(n, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for kw in (dict(t=0), dict(lr=-1.0), dict(clip=0.0), dict(clip=float("nan")),
                   dict(wd=float("inf"))):
            args = dict(t=1, lr=1e-3, wd=0.0, clip=1.0)
            args.update(kw)
            with pytest.raises(osr.AdamWError) as e:
                osr.adamw_clip_step(ctx, w, g, m, v, **args)
            assert e.value.status == osr.EINVAL
        with pytest.raises(osr.AdamWError) as e:
            osr.ckpt_pack(ctx, 1, w, m, v)
        assert e.value.status == osr.ESTATE


def test_80_step_trajectory_flat_65536(dev, oracle):
    """Configuration flat-65536: 80 steps with the clip active at every one;
    the GPU state against the oracle's own trajectory from the same inputs,
    every element, after step 1 (rtol 1e-6) and after every later step
    (rtol 1e-5, magnitudes carried along the trajectory)."""
    wl = W.flat_65k()
    n = wl.n
    (w, m, v), (ow, om, ov) = make_state(dev, n)
    idx = np.arange(n)
    run = Running()
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in range(1, wl.steps + 1):
            g, gh = grads(dev, n, wl, t)
            osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
            norm, scale = osr.adamw_last_norm(ctx)
            onorm = oracle.global_norm(gh)
            assert onorm > wl.clip and scale < 1.0
            assert abs(norm - onorm) <= RTOL_NORM * onorm
            s = oracle.clip_scale(onorm, wl.clip)
            terms = oracle.adamw_terms_at(idx, ow, gh, om, ov, s, t, wl.lr, wl.wd)
            mags = run.update(terms, wl.lr, wl.wd, t)
            oracle.adamw_clip_step(ow, gh, om, ov, t, wl.lr, wl.wd, wl.clip)
            rtol = RTOL_ONE_STEP if t == 1 else RTOL_TRAJECTORY
            assert_within(host(w, m, v), (ow, om, ov), mags, rtol, f"step {t}")


def _sampled_trajectory(dev, oracle, wl, steps, k=20_000, table=None, ckpt_dir=None):
    """GPU steps on the full state; the oracle follows k sampled elements
    exactly (its clip factor from its own norm of the full gradient).  With
    ckpt_dir, the final state is also packed and written, and the file is
    checked: exact size and header, its arrays equal to the GPU state, and
    its sampled values within the trajectory bar of the oracle."""
    n = wl.n
    (w, m, v), _ = make_state(dev, n, seed=wl.seed)
    g = torch.empty(n, device=dev)
    idx = sample_indices(n, k)
    idx_t = torch.from_numpy(idx).to(dev)

    def gathered():
        return [a[idx_t].cpu().numpy() for a in (w, m, v)]

    ow = synthetic.weights(wl.seed, idx=idx)  # the generator's values, drawn by index
    om = np.zeros(idx.size, np.float32)
    ov = np.zeros(idx.size, np.float32)
    assert ow.tobytes() == gathered()[0].tobytes()
    sub = np.arange(idx.size)
    run = Running()
    off, num = table if table else (None, None)
    flags = 0 if ckpt_dir else osr.CREATE_NO_CKPT
    with osr.adamw_create(n, off, num, flags=flags) as ctx:
        for t in range(1, steps + 1):
            synth_dev.fill_grads(g, wl.seed, t, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
            gh = g.cpu().numpy()
            osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
            norm, _ = osr.adamw_last_norm(ctx)
            onorm = oracle.global_norm(gh)
            assert abs(norm - onorm) <= RTOL_NORM * onorm, (t, norm, onorm)
            s = oracle.clip_scale(onorm, wl.clip)
            gs = gh[idx]
            terms = oracle.adamw_terms_at(sub, ow, gs, om, ov, s, t, wl.lr, wl.wd)
            mags = run.update(terms, wl.lr, wl.wd, t)
            ow, om, ov = oracle.adamw_at(sub, ow, gs, om, ov, s, t, wl.lr, wl.wd)
            if t == 1:
                assert_state_close(gathered(), (ow, om, ov), terms, RTOL_ONE_STEP, "step 1",
                                   lr=wl.lr, t=1)
        got = gathered()
        assert_within(got, (ow, om, ov), mags, RTOL_TRAJECTORY, f"after {steps} steps")
        if ckpt_dir:
            osr.ckpt_pack(ctx, steps, w, m, v, side_stream=torch.cuda.Stream())
            path = osr.ckpt_write(ctx, str(ckpt_dir))
            assert os.path.basename(path) == f"step_{steps:06d}.bin"
            assert os.path.getsize(path) == 8 + 12 * n
            with open(path, "rb") as f:
                assert struct.unpack("<ii", f.read(8)) == (steps, n)
            body = np.fromfile(path, dtype="<f4", offset=8)
            for r, a in enumerate((w, m, v)):
                assert body[r * n:(r + 1) * n].tobytes() == a.cpu().numpy().tobytes()
            from_file = [body[r * n + idx] for r in range(3)]
            assert_within(from_file, (ow, om, ov), mags, RTOL_TRAJECTORY, "file")


def test_flat_12m8_100_steps_writes_step_000100(dev, oracle, tmp_path):
    """Configuration flat-12.8M: 100 steps, then step_000100.bin of
    153,600,008 bytes; sampled elements against the oracle's trajectory."""
    wl = W.flat_12m8()
    _sampled_trajectory(dev, oracle, wl, wl.steps, ckpt_dir=tmp_path)
    assert osr.ckpt_file_size(wl.n) == 153_600_008


def test_gpt_110m_tensor_list_sampled(dev, oracle):
    wl = W.gpt_110m()
    _sampled_trajectory(dev, oracle, wl, 3, table=wl.table())


def test_flat_1b_one_step_sampled(dev, oracle):
    wl = W.flat_pow2(30)
    _sampled_trajectory(dev, oracle, wl, 1, k=50_000)
    torch.cuda.empty_cache()


def test_tensor_table_does_not_change_results(dev):
    """The offset table describes the flat layout; results are the flat
    vector's, bit for bit."""
    wl = W.gpt_110m()
    n = wl.n
    off, num = wl.table()
    outs = []
    for table in (None, (off, num)):
        (w, m, v), _ = make_state(dev, n)
        g = torch.empty(n, device=dev)
        o, k = table if table else (None, None)
        with osr.adamw_create(n, o, k, flags=osr.CREATE_NO_CKPT) as ctx:
            assert ctx.num_tensors == (196 if table else 1)
            for t in (1, 2):
                synth_dev.fill_grads(g, wl.seed, t, wl.grad_sigma)
                osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
            outs.append([x.cpu() for x in (w, m, v)])
        del w, m, v, g
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    torch.cuda.empty_cache()


def test_step_is_bit_stable(dev):
    n = 3_000_001
    res = []
    for _ in range(3):
        (w, m, v), _ = make_state(dev, n)
        g = torch.empty(n, device=dev)
        with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
            for t in range(1, 6):
                synth_dev.fill_grads(g, 7, t, 1e-2, 0.01, 100.0)
                osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
        res.append(torch.cat([w, m, v]).cpu())
    assert torch.equal(res[0], res[1]) and torch.equal(res[0], res[2])


@pytest.mark.parametrize("flags", [0, osr.LAUNCH_NO_ONEPASS])
def test_clip_threshold_is_strict(dev, flags):
    """g = [0.375, 0.5] has norm exactly 0.625 (exact squares and root).
    c = 0.625: no clip (the comparison is strict), factor exactly 1.
    c = 0.625 (1 - 2^-24): clipped, factor c / norm = 1 - 2^-24 exactly, the
    largest float below 1.  (One double below 0.625 also clips, but its
    factor 1 - 2^-53 rounds to 1.0f: the factor is a float.)"""
    g = torch.tensor([0.375, 0.5, 0.0, 0.0], device=dev)
    below = 0.625 * (1.0 - 2.0 ** -24)
    for clip, want_scale in ((0.625, 1.0), (below, float(np.float32(1.0 - 2.0 ** -24))),
                             (np.nextafter(0.625, 0.0), 1.0)):
        w = torch.tensor([1.0, -1.0, 0.5, 2.0], device=dev)
        m = torch.zeros(4, device=dev)
        v = torch.zeros(4, device=dev)
        with osr.adamw_create(4, flags=osr.CREATE_NO_CKPT) as ctx:
            osr.adamw_set_launch_options(ctx, flags)
            osr.adamw_clip_step(ctx, w, g, m, v, 1, 1e-3, 0.0, float(clip))
            norm, scale = osr.adamw_last_norm(ctx)
        assert norm == 0.625
        assert scale == want_scale, (clip, scale)
        # m = (1 - beta1) * (g s), one float32 rounding of each product
        gh = np.float32(np.float32(0.5) * np.float32(want_scale))
        assert m.cpu().numpy()[1] == np.float32(np.float32(0.1) * gh)


@pytest.mark.parametrize("which", ["gpt-110M-list", "flat-2^27+5"])
def test_dynamic_chunks_same_bits_as_static(dev, which):
    """The fused kernel hands chunks out by an atomic counter; every element
    is updated exactly once, so the whole state equals, bit for bit, the
    state after the same steps with chunks fixed per block (a skipped or
    repeated chunk would differ)."""
    n = W.gpt_110m().n if which == "gpt-110M-list" else (1 << 27) + 5
    outs = []
    for flags in (0, osr.LAUNCH_STATIC_CHUNKS):
        (w, m, v), _ = make_state(dev, n, m_sigma=1e-3, v_sigma=1e-5)
        g = torch.empty(n, device=dev)
        with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
            osr.adamw_set_launch_options(ctx, flags)
            for t in (1, 2, 3):
                synth_dev.fill_grads(g, 7, t, 1e-3, 0.001, 1000.0)
                osr.adamw_clip_step_ex(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0, zero_grad=(t == 3))
            torch.cuda.synchronize()
        outs.append([hashlib_digest(x) for x in (w, m, v, g)])
        del w, m, v, g
        torch.cuda.empty_cache()
    assert outs[0] == outs[1]


def hashlib_digest(t):
    import hashlib
    return hashlib.sha256(t.cpu().numpy().tobytes()).hexdigest()
