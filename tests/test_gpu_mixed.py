"""GPU mixed-precision step: bfloat16 / binary16 gradients and 16-bit weight
copies around float32 master weights and moments, against the oracle's mixed
step; the copy is the exact rounding of the GPU's own new weights and within
one 16-bit unit of the oracle's copy; zeroing, per-tensor sums and the
sharded sum of squares with 16-bit gradients; an 80-step trajectory."""
import numpy as np
import pytest

import synthetic
from parity import RTOL_NORM, RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, assert_within

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu
TORCH16 = {1: torch.bfloat16, 2: torch.float16}


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def bits16(x32, dt):
    return synthetic.to_bf16_bits(x32) if dt == 1 else synthetic.to_f16_bits(x32)


def decode(bits, dt):
    if dt == 1:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def upload16(bits, dt, dev):
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(TORCH16[dt])


def ulp16(x, dt):
    """Spacing of the 16-bit format at |x| (binary16 subnormals: 2^-24)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-45)))
    if dt == 1:
        return np.exp2(e - 7)
    return np.exp2(np.maximum(e, -14) - 10)


def check_copy(w_lp, w_gpu, w_lp_oracle, dt, w_oracle):
    """The copy is exactly the rounding of the GPU's own new weights, and
    differs from the oracle's copy by at most the weights' difference plus
    one 16-bit spacing (both round to nearest)."""
    lp = w_lp.view(torch.int16).cpu().numpy().view(np.uint16)
    assert lp.tobytes() == bits16(w_gpu, dt).tobytes()
    a = decode(lp, dt).astype(np.float64)
    b = decode(w_lp_oracle, dt).astype(np.float64)
    tol = (np.abs(w_gpu.astype(np.float64) - w_oracle)
           + ulp16(np.maximum(np.abs(w_gpu), np.abs(w_oracle)), dt))
    assert np.all(np.abs(a - b) <= tol)


@pytest.mark.parametrize("g_dt", [1, 2])
@pytest.mark.parametrize("lp_dt", [None, 1, 2])
def test_one_step(dev, oracle, g_dt, lp_dt):
    n = 1_000_003
    hw = synthetic.weights(7, n=n)
    hm = synthetic.draw(7, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(7, 12, 0, 1e-5, n=n))
    g32 = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    gb = bits16(g32, g_dt)
    w, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hm, hv))
    g = upload16(gb, g_dt, dev)
    w_lp = None if lp_dt is None else torch.empty(n, dtype=TORCH16[lp_dt], device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step_mixed(ctx, w, g, m, v, 1, 3e-3, 0.01, 1.0, w_lp=w_lp)
        norm, _ = osr.adamw_last_norm(ctx)
    ow, om, ov = hw.copy(), hm.copy(), hv.copy()
    _, onorm, olp = oracle.adamw_clip_step_mixed(ow, gb, g_dt, om, ov, 1, 3e-3, 0.01, 1.0,
                                                 w_lp_dtype=lp_dt)
    assert abs(norm - onorm) <= RTOL_NORM * onorm
    gd = decode(gb, g_dt)
    terms = oracle.adamw_terms_at(np.arange(n), hw, gd, hm, hv, oracle.clip_scale(onorm, 1.0),
                                  1, 3e-3, 0.01)
    mags = Running().update(terms, 3e-3, 0.01, 1)
    got = [x.cpu().numpy() for x in (w, m, v)]
    assert_within(got, (ow, om, ov), mags, RTOL_ONE_STEP, f"g={g_dt} lp={lp_dt}")
    if lp_dt is not None:
        check_copy(w_lp, got[0], olp, lp_dt, ow)


def test_zero_grad_tensor_norms_and_sumsq_16bit(dev, oracle):
    sizes = [24576, 1, 3, 768 * 7, 40000, 5]
    off = list(np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64))
    n = int(sum(sizes))
    g32 = synthetic.grads(7, 2, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    for dt in (1, 2):
        gb = bits16(g32, dt)
        gd = decode(gb, dt)
        g = upload16(gb, dt, dev)
        w, m, v = (torch.zeros(n, device=dev) for _ in range(3))
        with osr.adamw_create(n, off, sizes, flags=osr.CREATE_NO_CKPT) as ctx:
            s = osr.grad_sumsq_typed(ctx, g)
            want = oracle.sumsq(gd)
            assert abs(s - want) <= RTOL_NORM * want
            osr.adamw_clip_step_mixed(ctx, w, g, m, v, 1, 1e-3, 0.0, 1.0, zero_grad=True,
                                      tensor_norms=True)
            per = osr.adamw_last_tensor_sumsq(ctx)
            wantp = oracle.tensor_sumsq(gd, off, sizes)
            assert np.all(np.abs(per - wantp) <= RTOL_NORM * wantp)
        torch.cuda.synchronize()
        assert not bool(g.float().any())


def test_80_steps_bf16_grads_bf16_copy(dev, oracle):
    from synthetic import workloads as W
    wl = W.flat_65k()
    n = wl.n
    hw = synthetic.weights(wl.seed, n=n)
    w = torch.from_numpy(hw).to(dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    w_lp = torch.empty(n, dtype=torch.bfloat16, device=dev)
    ow, om, ov = hw.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    run = Running()
    idx = np.arange(n)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in range(1, wl.steps + 1):
            g32 = synthetic.grads(wl.seed, t, wl.grad_sigma, n=n, outlier_frac=wl.outlier_frac,
                                  outlier_mult=wl.outlier_mult)
            gb = bits16(g32, 1)
            osr.adamw_clip_step_mixed(ctx, w, upload16(gb, 1, dev), m, v, t, wl.lr, wl.wd,
                                      wl.clip, w_lp=w_lp)
            gd = decode(gb, 1)
            s = oracle.clip_scale(oracle.global_norm(gd), wl.clip)
            mags = run.update(oracle.adamw_terms_at(idx, ow, gd, om, ov, s, t, wl.lr, wl.wd),
                              wl.lr, wl.wd, t)
            _, _, olp = oracle.adamw_clip_step_mixed(ow, gb, 1, om, ov, t, wl.lr, wl.wd,
                                                     wl.clip, w_lp_dtype=1)
        got = [x.cpu().numpy() for x in (w, m, v)]
        assert_within(got, (ow, om, ov), mags, RTOL_TRAJECTORY, "after 80 steps")
        check_copy(w_lp, got[0], olp, 1, ow)


def test_misaligned_16bit_refused(dev):
    n = 1000
    w, m, v = (torch.zeros(n, device=dev) for _ in range(3))
    buf = torch.zeros(n + 4, dtype=torch.bfloat16, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        with pytest.raises(osr.AdamWError) as e:
            osr.adamw_clip_step_mixed(ctx, w, buf[1:n + 1], m, v, 1, 1e-3, 0.0, 1.0)
        assert e.value.status == osr.EINVAL


def test_full_size_bf16_copy_zero_grad_sampled(dev, oracle):
    """The 110M tensor list (chunks handed out by the counter at this size)
    with a bfloat16 gradient, a bfloat16 weight copy and zero_grad: the norm
    within 1e-6 of the oracle's, sampled elements within the one-step bar,
    the copy the exact rounding of the new weights there, and g zeroed."""
    from parity import assert_state_close, sample_indices
    from synthetic import device as synth_dev
    from synthetic import workloads as W
    wl = W.gpt_110m()
    n = wl.n
    off, num = wl.table()
    w = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    g32 = torch.empty(n, device=dev)
    synth_dev.fill_grads(g32, wl.seed, 1, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
    hw = w.cpu().numpy().copy()
    gb = bits16(g32.cpu().numpy(), 1)  # rounded on the host, uploaded as bits
    del g32
    g = upload16(gb, 1, dev)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    w_lp = torch.empty(n, dtype=torch.bfloat16, device=dev)
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step_mixed(ctx, w, g, m, v, 1, wl.lr, wl.wd, wl.clip, w_lp=w_lp,
                                  zero_grad=True)
        norm, _ = osr.adamw_last_norm(ctx)
    gd = decode(gb, 1)
    onorm = oracle.global_norm(gd)
    assert abs(norm - onorm) <= RTOL_NORM * onorm
    s = oracle.clip_scale(onorm, wl.clip)
    idx = sample_indices(n, 200_000)
    zeros = np.zeros(n, np.float32)
    want = oracle.adamw_at(idx, hw, gd, zeros, zeros, s, 1, wl.lr, wl.wd)
    terms = oracle.adamw_terms_at(idx, hw, gd, zeros, zeros, s, 1, wl.lr, wl.wd)
    ti = torch.from_numpy(idx).to(dev)
    got = [x[ti].cpu().numpy() for x in (w, m, v)]
    assert_state_close(got, want, terms, RTOL_ONE_STEP, "110M bf16", lr=wl.lr, t=1)
    lp = w_lp.view(torch.int16)[ti].cpu().numpy().view(np.uint16)
    assert lp.tobytes() == bits16(got[0], 1).tobytes()
    assert not bool(g.view(torch.int16).any())
