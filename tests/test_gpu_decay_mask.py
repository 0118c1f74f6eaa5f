"""GPU parity of the per-group weight decay (a decay flag per tensor of the
offset table; "Training as a Recoverable State Transition", section "The
Exact Targets of Clipping and AdamW": decaying every parameter is the
lesson's convention, not a claim about the best grouping).  The GPU step
with flags is compared with the oracle's masked step on the same generator
inputs: every element at ragged sizes, sampled elements on the 110M list, an
80-step trajectory, the unaligned scalar kernel, the 16-bit gradient path
and the step graph.  All calls go through the C ABI."""
import numpy as np
import pytest

import synthetic
from synthetic import workloads as W
from parity import (RTOL_NORM, RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, assert_within,
                    sample_indices)

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

LR, WD, CLIP = 3e-3, 0.1, 1.0  # a large wd, so that a flag slip is far outside tolerance


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def table(sizes):
    num = np.array(sizes, np.int64)
    off = np.concatenate([[0], np.cumsum(num)[:-1]]).astype(np.int64)
    return off, num


# ragged boundaries (not multiples of 4 or 32), runs of equal flags, a
# one-element tensor, exempt tensors at both ends
TABLES = {
    "ragged": ([3, 1000, 29, 4096, 1, 7, 33, 8192 * 3 + 5, 2, 31_000, 389],
               [0, 1, 0, 0, 1, 0, 1, 1, 0, 1, 0]),
    "one_exempt_middle": ([40_000, 1_237, 24_336], [1, 0, 1]),
    "all_exempt": ([65_573], [0]),
    "big_ragged": ([333_333, 3, 250_001, 16, 416_650], [0, 1, 1, 0, 1]),
}


def elem_flags(num, flags):
    return np.repeat(np.asarray(flags, bool), num)


def inputs(n, seed=7, m_sigma=1e-3, v_sigma=1e-5, g_sigma=1e-2, t=1):
    hw = synthetic.weights(seed, n=n)
    hm = synthetic.draw(seed, 11, 0, m_sigma, n=n)
    hv = np.abs(synthetic.draw(seed, 12, 0, v_sigma, n=n))
    hg = synthetic.grads(seed, t, g_sigma, n=n, outlier_frac=0.01, outlier_mult=100.0)
    return hw, hg, hm, hv


def masked_terms(oracle, idx, w, g, m, v, s, t, lr, wd, eflags):
    """The oracle's double terms at idx, each with its own tensor's wd."""
    on = oracle.adamw_terms_at(idx, w, g, m, v, s, t, lr, wd)
    off = oracle.adamw_terms_at(idx, w, g, m, v, s, t, lr, 0.0)
    return np.where(eflags[idx][:, None], on, off)


def check_one_step(oracle, got, hw, hg, hm, hv, off, num, flags, t, lr=LR, wd=WD, label=""):
    ow, om, ov = hw.copy(), hm.copy(), hv.copy()
    _, onorm = oracle.adamw_clip_step_masked(ow, hg, om, ov, off, num, flags, t, lr, wd, CLIP)
    ef = elem_flags(num, flags)
    idx = np.arange(hw.size)
    terms = masked_terms(oracle, idx, hw, hg, hm, hv, oracle.clip_scale(onorm, CLIP), t, lr,
                         wd, ef)
    mags = Running().update(terms, lr, np.where(ef, wd, 0.0), t)
    assert_within(got, (ow, om, ov), mags, RTOL_ONE_STEP, label)
    return onorm


@pytest.mark.parametrize("name", sorted(TABLES))
def test_one_step_all_elements(dev, oracle, name):
    sizes, flags = TABLES[name]
    off, num = table(sizes)
    n = int(num.sum())
    for t in (1, 7):
        hw, hg, hm, hv = inputs(n, t=t)
        w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
        with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
            osr.adamw_set_decay_mask(ctx, flags)
            osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            norm, _ = osr.adamw_last_norm(ctx)
        got = [x.cpu().numpy() for x in (w, m, v)]
        onorm = check_one_step(oracle, got, hw, hg, hm, hv, off, num, flags, t,
                               label=f"{name} t={t}")
        assert abs(norm - onorm) <= RTOL_NORM * onorm


def test_exempt_weights_with_zero_gradient_stay_exact(dev):
    """A zero gradient leaves an exempt weight bit for bit as it was (its
    decay factor is exactly 1 and its update exactly 0), and moves every
    flagged one."""
    sizes, flags = TABLES["ragged"]
    off, num = table(sizes)
    n = int(num.sum())
    hw = synthetic.weights(7, n=n)
    w = torch.from_numpy(hw).to(dev)
    g, m, v = (torch.zeros(n, device=dev) for _ in range(3))
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_decay_mask(ctx, flags)
        osr.adamw_clip_step(ctx, w, g, m, v, 1, LR, WD, CLIP)
        torch.cuda.synchronize()
    got = w.cpu().numpy()
    ef = elem_flags(num, flags)
    assert got[~ef].tobytes() == hw[~ef].tobytes()
    moved = got[ef] != hw[ef]
    assert moved[hw[ef] != 0].all()


def test_all_flags_and_clearing_give_the_default_bits(dev):
    """All flags set, or the flags cleared again, is the unmasked step bit
    for bit."""
    sizes, flags = TABLES["big_ragged"]
    off, num = table(sizes)
    n = int(num.sum())
    hw, hg, hm, hv = inputs(n)
    outs = {}
    for mode in ("default", "all_set", "cleared"):
        w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
        with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
            if mode == "all_set":
                osr.adamw_set_decay_mask(ctx, [1] * len(sizes))
            elif mode == "cleared":
                osr.adamw_set_decay_mask(ctx, flags)
                osr.adamw_set_decay_mask(ctx, None)
            for t in (1, 2, 3):
                osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            torch.cuda.synchronize()
        outs[mode] = [x.cpu().numpy().tobytes() for x in (w, m, v)]
    assert outs["all_set"] == outs["default"]
    assert outs["cleared"] == outs["default"]


def test_80_step_trajectory(dev, oracle):
    """80 steps of the flat-65536 kind of input (1% outliers x100, the clip
    on at every step) under the ragged grouping; every element against the
    oracle's masked trajectory after each step."""
    sizes, flags = TABLES["ragged"]
    off, num = table(sizes)
    n = int(num.sum())
    ef = elem_flags(num, flags)
    wd_e = np.where(ef, WD, 0.0)
    hw = synthetic.weights(7, n=n)
    ow, om, ov = hw.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    w = torch.from_numpy(hw).to(dev)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    idx = np.arange(n)
    run = Running()
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_decay_mask(ctx, flags)
        for t in range(1, 81):
            hg = synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
            osr.adamw_clip_step(ctx, w, torch.from_numpy(hg).to(dev), m, v, t, LR, WD, CLIP)
            norm, _ = osr.adamw_last_norm(ctx)
            s = oracle.clip_scale(oracle.global_norm(hg), CLIP)
            terms = masked_terms(oracle, idx, ow, hg, om, ov, s, t, LR, WD, ef)
            mags = run.update(terms, LR, wd_e, t)
            _, onorm = oracle.adamw_clip_step_masked(ow, hg, om, ov, off, num, flags, t, LR,
                                                     WD, CLIP)
            assert abs(norm - onorm) <= RTOL_NORM * onorm
            got = [x.cpu().numpy() for x in (w, m, v)]
            assert_within(got, (ow, om, ov), mags,
                          RTOL_ONE_STEP if t == 1 else RTOL_TRAJECTORY, f"t={t}")


def test_gpt_110m_matrices_only_sampled(dev, oracle):
    """The 110M tensor list with decay on matrices and embeddings only
    (biases and norm parameters exempt): the norm, and sampled elements of
    every tensor kind against the oracle one by one."""
    wl = W.gpt_110m()
    off, num = (np.array(x, np.int64) for x in wl.table())
    flags = W.decay_flags_matrices_only(wl.tensors)
    assert 0 < sum(flags) < len(flags)
    n = wl.n
    ef = elem_flags(num, flags)
    from synthetic import device as synth_dev
    w, g = torch.empty(n, device=dev), torch.empty(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    synth_dev.fill_grads(g, wl.seed, 1, wl.grad_sigma)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    hw, hg = w.cpu().numpy(), g.cpu().numpy()
    assert hw[:1000].tobytes() == synthetic.weights(wl.seed, n=1000).tobytes()
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_decay_mask(ctx, flags)
        osr.adamw_clip_step(ctx, w, g, m, v, 1, LR, WD, CLIP)
        norm, _ = osr.adamw_last_norm(ctx)
    onorm = oracle.global_norm(hg)
    assert abs(norm - onorm) <= RTOL_NORM * onorm
    # every tensor's first and last element, plus the usual sample
    idx = np.unique(np.concatenate([off, off + num - 1, sample_indices(n, 200_000)]))
    z = np.zeros(n, np.float32)
    s = oracle.clip_scale(onorm, CLIP)
    terms = masked_terms(oracle, idx, hw, hg, z, z, s, 1, LR, WD, ef)
    wa, ma, va = oracle.adamw_at(idx, hw, hg, z, z, s, 1, LR, WD)
    wb, mb, vb = oracle.adamw_at(idx, hw, hg, z, z, s, 1, LR, 0.0)
    sel = ef[idx]
    want = (np.where(sel, wa, wb), ma, va)
    mags = Running().update(terms, LR, np.where(sel, WD, 0.0), 1)
    got = [x[torch.from_numpy(idx).to(dev)].cpu().numpy() for x in (w, m, v)]
    assert_within(got, want, mags, RTOL_ONE_STEP, "gpt-110M matrices-only")


def test_unaligned_views_take_the_scalar_kernel(dev, oracle):
    sizes, flags = TABLES["ragged"]
    off, num = table(sizes)
    n = int(num.sum())
    hw, hg, hm, hv = inputs(n)
    bufs = [torch.empty(n + 1, device=dev) for _ in range(4)]
    w, g, m, v = (b[1:] for b in bufs)
    assert all(x.data_ptr() % 16 == 4 for x in (w, g, m, v))
    for d, h in zip((w, g, m, v), (hw, hg, hm, hv)):
        d.copy_(torch.from_numpy(h))
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_decay_mask(ctx, flags)
        osr.adamw_clip_step(ctx, w, g, m, v, 2, LR, WD, CLIP)
    got = [x.cpu().numpy() for x in (w, m, v)]
    check_one_step(oracle, got, hw, hg, hm, hv, off, num, flags, 2, label="unaligned")


def test_bf16_gradient_path(dev, oracle):
    """The 16-bit gradient kernels apply the same flags (bfloat16 gradients
    that are exact in bfloat16, so the oracle's float32 masked step is the
    reference)."""
    sizes, flags = TABLES["big_ragged"]
    off, num = table(sizes)
    n = int(num.sum())
    hw, hg32, hm, hv = inputs(n)
    bits = synthetic.to_bf16_bits(hg32)
    hg = (bits.astype(np.uint32) << 16).view(np.float32)  # exact widening
    g = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    w, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hm, hv))
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_decay_mask(ctx, flags)
        osr.adamw_clip_step_mixed(ctx, w, g, m, v, 1, LR, WD, CLIP)
    got = [x.cpu().numpy() for x in (w, m, v)]
    check_one_step(oracle, got, hw, hg, hm, hv, off, num, flags, 1, label="bf16")


def test_graph_step_applies_the_flags(dev):
    """The step graph reads the same flags, and setting or clearing them
    after the graph was made takes effect at the next graph step: bit for
    bit the plain steps through the same sequence."""
    sizes, flags = TABLES["big_ragged"]
    off, num = table(sizes)
    n = int(num.sum())
    hw, hg, hm, hv = inputs(n)
    plan = {1: None, 2: flags, 3: None, 4: None, 5: [1 - f for f in flags], 6: None}
    outs = []
    for use_graph in (False, True):
        w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
        with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
            if use_graph:
                osr.adamw_graph_create(ctx, w, g, m, v)
            for t in range(1, 7):
                if t in (2, 4, 5):
                    osr.adamw_set_decay_mask(ctx, plan[t])
                if use_graph:
                    osr.adamw_graph_step(ctx, t, LR, WD, CLIP)
                else:
                    osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            torch.cuda.synchronize()
            if use_graph:
                osr.adamw_graph_destroy(ctx)
        outs.append([x.cpu().numpy().tobytes() for x in (w, m, v)])
    assert outs[0] == outs[1]


def test_bad_arguments(dev):
    off, num = table([10, 20, 30])
    with osr.adamw_create(60, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        with pytest.raises(osr.AdamWError) as e:
            osr.adamw_set_decay_mask(ctx, [1, 0])
        assert e.value.status == osr.EINVAL
        osr.adamw_set_decay_mask(ctx, [1, 0, 1])
        osr.adamw_set_decay_mask(ctx, None)
