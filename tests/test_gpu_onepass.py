"""The one-launch step (small states: norm, clip factor and update in one
cooperative grid) against the two-launch step: the same bits for w, m, v, g
and the norm, with and without decay flags, zero-grad and a gradient scale;
its bounded grid-barrier wait runs out cleanly when made to wait for a block
that does not exist.  Oracle parity of the default path at these sizes is
covered by the other GPU tests, which now take this path."""
import numpy as np
import pytest

import synthetic

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

LR, WD, CLIP = 3e-3, 0.05, 1.0


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def inputs(n, seed=7):
    hw = synthetic.weights(seed, n=n)
    hm = synthetic.draw(seed, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(seed, 12, 0, 1e-5, n=n))
    return hw, hm, hv


def run(dev, n, launch_flags, steps=4, mask=None, zero_grad=False, grad_scale=1.0, table=None):
    hw, hm, hv = inputs(n)
    w, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hm, hv))
    norms, grads = [], []
    off, num = table if table is not None else (None, None)
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_launch_options(ctx, launch_flags)
        if mask is not None:
            osr.adamw_set_decay_mask(ctx, mask)
        for t in range(1, steps + 1):
            hg = synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
            g = torch.from_numpy(hg).to(dev)
            osr.adamw_clip_step_ex(ctx, w, g, m, v, t, LR, WD, CLIP, grad_scale=grad_scale,
                                   zero_grad=zero_grad)
            norms.append(osr.adamw_last_norm(ctx))
            grads.append(g.cpu().numpy().tobytes())
    return [x.cpu().numpy().tobytes() for x in (w, m, v)], norms, grads


@pytest.mark.parametrize("n", [1, 3, 4, 5, 4093, 8191, 8192, 8193, 65536, 65573, 100_003,
                               (1 << 19) - 4, 1 << 19])
def test_same_bits_as_two_launches(dev, n):
    a = run(dev, n, 0)
    b = run(dev, n, osr.LAUNCH_NO_ONEPASS)
    assert a[0] == b[0]
    assert a[1] == b[1]  # norm (double) and factor (float), bit for bit
    assert a[2] == b[2]


@pytest.mark.parametrize("last", [24_533, 24_496])
def test_same_bits_with_flags_zero_grad_and_scale(dev, last):
    """65,573 parameters: the cooperative grid; 65,536: a cluster size, where
    zero_grad takes the grid form (the cluster form never zeroes g)."""
    sizes = [3, 1000, 29, 40_000, 1, 7, last]
    num = np.array(sizes, np.int64)
    off = np.concatenate([[0], np.cumsum(num)[:-1]]).astype(np.int64)
    n = int(num.sum())
    mask = [1, 0, 1, 1, 0, 0, 1]
    kw = dict(mask=mask, zero_grad=True, grad_scale=0.25, table=(off, num))
    a = run(dev, n, 0, **kw)
    b = run(dev, n, osr.LAUNCH_NO_ONEPASS, **kw)
    assert a == b
    assert all(gb == bytes(4 * n) for gb in a[2])  # zero_grad wrote zeros


@pytest.mark.parametrize("n", [40_000, 65_573])
def test_barrier_timeout_is_reported_and_the_context_recovers(dev, n):
    """Made to wait for one block more than it launched, the grid's bounded
    wait runs out (about a second): the step is skipped, adamw_last_norm
    reports ADAMW_ECUDA once, and the next steps match a run that never
    faulted.  At 40,000 parameters the test flag takes the cooperative grid
    and the step after it the cluster form."""
    hw, hm, hv = inputs(n)
    w, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hm, hv))
    g = torch.from_numpy(synthetic.grads(7, 1, 1e-2, n=n)).to(dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_launch_options(ctx, osr.LAUNCH_TEST_BARRIER_TIMEOUT)
        osr.adamw_clip_step(ctx, w, g, m, v, 1, LR, WD, CLIP)
        with pytest.raises(osr.AdamWError) as e:
            osr.adamw_last_norm(ctx)
        assert e.value.status == osr.ECUDA and "barrier" in str(e.value)
        for d, h in zip((w, m, v), (hw, hm, hv)):
            assert d.cpu().numpy().tobytes() == h.tobytes()  # nothing was updated
        # the flag was one-shot and the fault is cleared once reported
        osr.adamw_clip_step(ctx, w, g, m, v, 1, LR, WD, CLIP)
        got_norm = osr.adamw_last_norm(ctx)
        got = [x.cpu().numpy().tobytes() for x in (w, m, v)]
    w2, m2, v2 = (torch.from_numpy(x).to(dev) for x in (hw, hm, hv))
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_ONEPASS)
        osr.adamw_clip_step(ctx, w2, g, m2, v2, 1, LR, WD, CLIP)
        assert osr.adamw_last_norm(ctx) == got_norm
    assert got == [x.cpu().numpy().tobytes() for x in (w2, m2, v2)]


def test_large_or_unaligned_states_take_two_launches(dev):
    """The test flag only affects the one-launch path: above 2^19 parameters
    and for unaligned arrays the step runs as two launches and does not
    fault."""
    for n, offset in (((1 << 19) + 4, 0), (50_000, 1)):
        bufs = [torch.zeros(n + offset, device=dev) for _ in range(4)]
        w, g, m, v = (b[offset:] for b in bufs)
        g.fill_(1e-3)
        with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
            osr.adamw_set_launch_options(ctx, osr.LAUNCH_TEST_BARRIER_TIMEOUT)
            osr.adamw_clip_step(ctx, w, g, m, v, 1, LR, WD, CLIP)
            osr.adamw_last_norm(ctx)


@pytest.mark.parametrize("n", [40_003, 65_573])
def test_captured_steps_match_eager_two_launch_steps(dev, n):
    """Steps captured into a graph replay to the bits of eager two-launch
    steps: at 40,003 parameters each step is one cluster-kernel node; at
    65,573 (above the cluster form) captured steps are two kernel nodes,
    which take less GPU time there than the cooperative grid."""
    hw, hm, hv = inputs(n)
    hg = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    a = [torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv)]
    b = [torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv)]
    ctx_a = osr.adamw_create(n, flags=osr.CREATE_NO_CKPT)
    ctx_b = osr.adamw_create(n, flags=osr.CREATE_NO_CKPT)
    osr.adamw_set_launch_options(ctx_a, osr.LAUNCH_NO_ONEPASS)
    cap = torch.cuda.Stream()
    gr = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gr, stream=cap):
            for t in (3, 4):
                osr.adamw_clip_step(ctx_b, b[0], b[1], b[2], b[3], t, LR, WD, CLIP, stream=cap)
    for _ in range(3):
        gr.replay()
        for t in (3, 4):
            osr.adamw_clip_step(ctx_a, a[0], a[1], a[2], a[3], t, LR, WD, CLIP)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    del gr
    ctx_a.close()
    ctx_b.close()


def test_step_graph_one_node_matches_plain_steps(dev):
    """The library's step graph up to 65,536 parameters is one cluster node;
    through a sequence that sets decay flags, switches the one-launch step
    off and on again (each change rebuilds the graph), its steps equal plain
    two-launch steps bit for bit."""
    sizes = [1000, 3, 59_992, 5, 4_536]
    num = np.array(sizes, np.int64)
    off = np.concatenate([[0], np.cumsum(num)[:-1]]).astype(np.int64)
    n = int(num.sum())
    hw, hm, hv = inputs(n)
    hg = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    plan = {2: ("mask", [1, 0, 1, 1, 0]), 4: ("opts", osr.LAUNCH_NO_ONEPASS), 5: ("opts", 0),
            6: ("mask", None)}
    outs, norms = [], []
    for use_graph in (False, True):
        w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
        got_norms = []
        with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
            if not use_graph:
                osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_ONEPASS)
            else:
                osr.adamw_graph_create(ctx, w, g, m, v)
            for t in range(1, 8):
                kind, val = plan.get(t, (None, None))
                if kind == "mask":
                    osr.adamw_set_decay_mask(ctx, val)
                elif kind == "opts" and use_graph:
                    osr.adamw_set_launch_options(ctx, val)
                if use_graph:
                    osr.adamw_graph_step(ctx, t, LR, WD, CLIP)
                else:
                    osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
                got_norms.append(osr.adamw_last_norm(ctx))
            if use_graph:
                osr.adamw_graph_destroy(ctx)
        outs.append([x.cpu().numpy().tobytes() for x in (w, m, v)])
        norms.append(got_norms)
    assert outs[0] == outs[1]
    assert norms[0] == norms[1]


def test_step_graph_barrier_timeout_is_reported(dev):
    """Above 65,536 parameters the step graph has two nodes; the test flag
    makes its next step rebuild it around the cooperative grid, whose
    barrier then runs out, and the step after that rebuilds the two nodes."""
    n = 100_003
    hw, hm, hv = inputs(n)
    w, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hm, hv))
    g = torch.from_numpy(synthetic.grads(7, 1, 1e-2, n=n)).to(dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_graph_create(ctx, w, g, m, v)
        osr.adamw_set_launch_options(ctx, osr.LAUNCH_TEST_BARRIER_TIMEOUT)
        osr.adamw_graph_step(ctx, 1, LR, WD, CLIP)
        with pytest.raises(osr.AdamWError) as e:
            osr.adamw_last_norm(ctx)
        assert e.value.status == osr.ECUDA
        for d, h in zip((w, m, v), (hw, hm, hv)):
            assert d.cpu().numpy().tobytes() == h.tobytes()
        osr.adamw_graph_step(ctx, 1, LR, WD, CLIP)
        osr.adamw_last_norm(ctx)
        assert not torch.equal(w, torch.from_numpy(hw).to(dev))
        osr.adamw_graph_destroy(ctx)


def test_cluster_step_graph_ignores_the_timeout_flag(dev):
    """Up to 65,536 parameters the graph's node is the cluster kernel, which
    has no software barrier: the test flag is consumed and the step runs
    normally, with the two-launch step's bits."""
    n = 40_000
    hw, hm, hv = inputs(n)
    hg = synthetic.grads(7, 1, 1e-2, n=n)
    w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_graph_create(ctx, w, g, m, v)
        osr.adamw_set_launch_options(ctx, osr.LAUNCH_TEST_BARRIER_TIMEOUT)
        osr.adamw_graph_step(ctx, 1, LR, WD, CLIP)
        got_norm = osr.adamw_last_norm(ctx)
        got = [x.cpu().numpy().tobytes() for x in (w, m, v)]
    w2, g2, m2, v2 = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_ONEPASS)
        osr.adamw_clip_step(ctx, w2, g2, m2, v2, 1, LR, WD, CLIP)
        assert osr.adamw_last_norm(ctx) == got_norm
    assert got == [x.cpu().numpy().tobytes() for x in (w2, m2, v2)]


@pytest.mark.parametrize("sizes", [[3, 1000, 29, 40_000, 1, 7, 24_496], [5, 39_998]])
def test_cluster_form_with_flags_same_bits(dev, sizes):
    """The cluster form (no zero_grad) with decay flags, a gradient scale and
    a ragged n % 4 tail, eager and in the step graph, against two launches."""
    num = np.array(sizes, np.int64)
    off = np.concatenate([[0], np.cumsum(num)[:-1]]).astype(np.int64)
    n = int(num.sum())
    mask = [k % 2 for k in range(len(sizes))]
    kw = dict(mask=mask, grad_scale=0.25, table=(off, num))
    a = run(dev, n, 0, **kw)
    b = run(dev, n, osr.LAUNCH_NO_ONEPASS, **kw)
    assert a == b
    hw, hm, hv = inputs(n)
    hg = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    outs = []
    for use_graph in (False, True):
        w, g, m, v = (torch.from_numpy(x).to(dev) for x in (hw, hg, hm, hv))
        with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
            osr.adamw_set_decay_mask(ctx, mask)
            if use_graph:
                osr.adamw_graph_create(ctx, w, g, m, v)
            else:
                osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_ONEPASS)
            for t in range(1, 4):
                if use_graph:
                    osr.adamw_graph_step(ctx, t, LR, WD, CLIP)
                else:
                    osr.adamw_clip_step(ctx, w, g, m, v, t, LR, WD, CLIP)
            outs.append(([x.cpu().numpy().tobytes() for x in (w, m, v)],
                         osr.adamw_last_norm(ctx)))
    assert outs[0] == outs[1]
