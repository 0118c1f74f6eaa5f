"""The sharded step with the exchange on the device (grad_sumsq_to, an
all-gather, adamw_clip_step_gathered) against the host-side exchange
(grad_sumsq, the gathered values handed to adamw_clip_step_ranks, which
adds them in rank order on the host): the same bits, for 1 to 4 virtual ranks on one GPU (each rank
one context over its shard; the all-gather is a copy of each rank's value
into its slot).  Also: a single rank equals the plain step, and a non-finite
gradient on one rank skips every rank's update."""
import numpy as np
import pytest

import synthetic
from optimizer_step_resumable_gb300 import sharded

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

LR, WD, CLIP = 3e-3, 0.01, 1.0


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def shards(dev, n, world):
    hw = synthetic.weights(7, n=n)
    hm = synthetic.draw(7, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(7, 12, 0, 1e-5, n=n))
    out = []
    for r in range(world):
        off, num = sharded.shard_range(n, r, world)
        out.append((off, num, [torch.from_numpy(x[off:off + num].copy()).to(dev)
                               for x in (hw, hm, hv)]))
    return out


# every world size at both sizes for a float32 gradient; one size suffices
# for the 16-bit gradient; one shard of 2^24 + 5 parameters takes the
# counter-scheduled chunks behind both exchanges
CASES = ([(w, n, "f32") for w in (1, 2, 3, 4) for n in (65_573, 1_000_003)] +
         [(w, 1_000_003, "bf16") for w in (1, 2, 3, 4)] + [(1, (1 << 24) + 5, "f32")])


@pytest.mark.parametrize("world,n,gdt", CASES)
def test_device_exchange_same_bits_as_host_exchange(dev, world, n, gdt):
    runs = []
    for mode in ("host", "device"):
        parts = shards(dev, n, world)
        ctxs = [osr.adamw_create(num, flags=osr.CREATE_NO_CKPT) for _, num, _ in parts]
        recv = torch.zeros(world, dtype=torch.float64, device=dev)
        norms = []
        for t in (1, 2, 3):
            hg = synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
            gs = [torch.from_numpy(hg[off:off + num].copy()).to(dev) for off, num, _ in parts]
            if gdt == "bf16":
                gs = [g.to(torch.bfloat16) for g in gs]
            if mode == "host":
                sums = [osr.grad_sumsq_typed(c, g) for c, g in zip(ctxs, gs)]
                for c, (_, _, (w, m, v)), g in zip(ctxs, parts, gs):
                    osr.adamw_clip_step_ranks(c, w, g, m, v, t, LR, WD, CLIP, sums)
            else:
                for r, (c, g) in enumerate(zip(ctxs, gs)):
                    osr.grad_sumsq_to(c, g, recv[r:r + 1])
                for c, (_, _, (w, m, v)), g in zip(ctxs, parts, gs):
                    osr.adamw_clip_step_gathered(c, w, g, m, v, t, LR, WD, CLIP, recv)
                norms.append([osr.adamw_last_norm(c) for c in ctxs])
        torch.cuda.synchronize()
        runs.append([x.cpu().numpy().tobytes() for _, _, xs in parts for x in xs])
        if mode == "device":
            # every rank published the same global norm
            for per_rank in norms:
                assert all(x == per_rank[0] for x in per_rank)
        for c in ctxs:
            c.close()
    assert runs[0] == runs[1]


def test_single_rank_equals_the_plain_step(dev):
    n = 100_003
    (_, _, a), = shards(dev, n, 1)
    (_, _, b), = shards(dev, n, 1)
    hg = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    g = torch.from_numpy(hg).to(dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ca, \
            osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as cb:
        osr.adamw_set_launch_options(ca, osr.LAUNCH_NO_ONEPASS)
        osr.adamw_clip_step(ca, *a[:1], g, *a[1:], 1, LR, WD, CLIP)
        ex = sharded.DeviceExchange(1, dev)
        sharded.sharded_clip_step_device(cb, b[0], g, b[1], b[2], 1, LR, WD, CLIP, ex)
        assert osr.adamw_last_norm(ca) == osr.adamw_last_norm(cb)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_nonfinite_on_one_rank_skips_every_rank(dev):
    n, world = 40_000, 3
    parts = shards(dev, n, world)
    before = [[x.clone() for x in xs] for _, _, xs in parts]
    ctxs = [osr.adamw_create(num, flags=osr.CREATE_NO_CKPT) for _, num, _ in parts]
    recv = torch.zeros(world, dtype=torch.float64, device=dev)
    gs = [torch.full((num,), 1e-3, device=dev) for _, num, _ in parts]
    gs[1][17] = float("inf")
    for r, (c, g) in enumerate(zip(ctxs, gs)):
        osr.grad_sumsq_to(c, g, recv[r:r + 1])
    for c, (_, _, (w, m, v)), g in zip(ctxs, parts, gs):
        osr.adamw_clip_step_gathered(c, w, g, m, v, 1, LR, WD, CLIP, recv)
    for c in ctxs:
        with pytest.raises(osr.NonFiniteGradient):
            osr.adamw_last_norm(c)
    for (_, _, xs), bs in zip(parts, before):
        for x, b in zip(xs, bs):
            assert torch.equal(x, b)
    for c in ctxs:
        c.close()


def test_bad_arguments(dev):
    n = 1000
    w, g, m, v = (torch.zeros(n, device=dev) for _ in range(4))
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        with pytest.raises(ValueError):
            osr.grad_sumsq_to(ctx, g, torch.zeros(1, device=dev))  # float32, not float64
        empty = torch.zeros(0, dtype=torch.float64, device=dev)
        with pytest.raises((ValueError, osr.AdamWError)):
            osr.adamw_clip_step_gathered(ctx, w, g, m, v, 1, LR, WD, CLIP, empty)
