"""GPU: the sharded step on R virtual shards of one GPU (each shard its own
context, sums of squares exchanged in rank order), gradient accumulation with
the 1/k scale folded into the clip factor, and the fused zero_grads."""
import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from parity import RTOL_NORM, RTOL_ONE_STEP, RTOL_TRAJECTORY, Running, assert_within

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402
from optimizer_step_resumable_gb300.sharded import shard_range  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_virtual_shards_match_oracle(dev, oracle, world):
    """R ranks emulated as R contexts over R contiguous shards of one state:
    3 steps, every element against the oracle's unsharded trajectory."""
    n = 1_000_003
    hw = synthetic.weights(7, n=n)
    w = torch.from_numpy(hw).to(dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    ow, om, ov = hw.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    spans = [shard_range(n, r, world) for r in range(world)]
    ctxs = [osr.adamw_create(k, flags=osr.CREATE_NO_CKPT) for _, k in spans]
    run = Running()
    idx = np.arange(n)
    try:
        for t in (1, 2, 3):
            hg = synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
            g = torch.from_numpy(hg).to(dev)
            sl = [slice(o, o + k) for o, k in spans]
            parts = [osr.grad_sumsq(c, g[s]) for c, s in zip(ctxs, sl)]
            total = osr.adamw_rank_total(parts, 1.0)[0]
            for c, s in zip(ctxs, sl):
                osr.adamw_clip_step_ranks(c, w[s], g[s], m[s], v[s], t, 3e-3, 0.01, 1.0, parts)
            onorm = oracle.global_norm(hg)
            assert abs(np.sqrt(total) - onorm) <= RTOL_NORM * onorm
            s_or = oracle.clip_scale(onorm, 1.0)
            mags = run.update(oracle.adamw_terms_at(idx, ow, hg, om, ov, s_or, t, 3e-3, 0.01),
                              3e-3, 0.01, t)
            oracle.adamw_clip_step(ow, hg, om, ov, t, 3e-3, 0.01, 1.0)
            got = [x.cpu().numpy() for x in (w, m, v)]
            assert_within(got, (ow, om, ov), mags, RTOL_ONE_STEP if t == 1 else RTOL_TRAJECTORY,
                          f"world={world} t={t}")
    finally:
        for c in ctxs:
            c.close()


def test_global_sumsq_nonfinite_skips_without_launch(dev):
    n = 1000
    w = torch.ones(n, device=dev)
    g = torch.ones(n, device=dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for bad in (float("inf"), float("nan")):
            with pytest.raises(osr.NonFiniteGradient):
                osr.adamw_clip_step_ex(ctx, w, g, m, v, 1, 1e-3, 0.0, 1.0, global_sumsq=bad)
        torch.cuda.synchronize()
        assert bool((w == 1).all()) and not bool(m.any())


def test_micro_batch_accumulation_and_zero_grad(dev, oracle):
    """backward adds 4 micro-batch gradients into one buffer; the step with
    grad_scale 1/4 and ZERO_GRAD equals the oracle's step on the scaled
    buffer and leaves the buffer zeroed for the next accumulation."""
    n = 2_000_003
    k = 4
    hw = synthetic.weights(7, n=n)
    w = torch.from_numpy(hw).to(dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    g = torch.zeros(n, device=dev)
    ow, om, ov = hw.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    run = Running()
    idx = np.arange(n)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in (1, 2):
            acc = np.zeros(n, np.float32)
            for j in range(k):  # same float32 adds, same order, on both sides
                part = synthetic.draw(7, 20 + j, t, 1e-2, n=n)
                g += torch.from_numpy(part).to(dev)
                acc += part
            assert g.cpu().numpy().tobytes() == acc.tobytes()
            osr.adamw_clip_step_ex(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0, grad_scale=1.0 / k,
                                   zero_grad=True)
            norm, _ = osr.adamw_last_norm(ctx)
            _, onorm = oracle.adamw_clip_step_scaled(ow.copy(), acc, om.copy(), ov.copy(), t,
                                                     3e-3, 0.01, 1.0, 1.0 / k)
            assert abs(norm - onorm) <= RTOL_NORM * onorm
            s = oracle.clip_scale(onorm, 1.0)

            terms = oracle.adamw_terms_at(idx, ow, acc, om, ov, s / k, t, 3e-3, 0.01)
            mags = run.update(terms, 3e-3, 0.01, t)
            oracle.adamw_clip_step_scaled(ow, acc, om, ov, t, 3e-3, 0.01, 1.0, 1.0 / k)
            got = [x.cpu().numpy() for x in (w, m, v)]
            assert_within(got, (ow, om, ov), mags, RTOL_ONE_STEP if t == 1 else RTOL_TRAJECTORY,
                          f"t={t}")
            assert not bool(g.any())  # zeroed by the fused kernel



def test_zero_grad_scalar_path_and_tail(dev):
    """The zeroing also covers the unaligned kernel and the ragged tail."""
    for n, off in ((4099, 0), (4099, 1)):
        buf = torch.empty(n + 1, device=dev)
        g = buf[off:off + n]
        synth_dev.fill_grads(g, 7, 1, 1e-2)
        w, m, v = (torch.zeros(n, device=dev) for _ in range(3))
        with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
            osr.adamw_clip_step_ex(ctx, w, g, m, v, 1, 1e-3, 0.0, 1.0, zero_grad=True)
        torch.cuda.synchronize()
        assert not bool(g.any()) and bool(m.any())
