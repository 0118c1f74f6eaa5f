"""GPU: the step graph gives the same bits as the plain two-launch step,
with per-step scalars (t, lr, clip) rewritten into the instantiated graph."""
import pytest

from synthetic import device as synth_dev

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _state(dev, n, offset=0):
    bufs = [torch.empty(n + offset, device=dev) for _ in range(4)]
    w, g, m, v = (b[offset:] for b in bufs)
    synth_dev.fill_weights(w, 7)
    m.zero_()
    v.zero_()
    return w, g, m, v


@pytest.mark.parametrize("n,offset", [(65536, 0), (1_000_003, 0), (40_001, 1),
                                      ((1 << 24) + 5, 0)])
def test_graph_steps_equal_plain_steps(dev, n, offset):
    """(2^24 + 5: the fused node hands chunks out by its counter, which must
    reset itself for every replay.)"""
    a = _state(dev, n, offset)
    b = _state(dev, n, offset)
    sched = [(t, 3e-3 * (0.5 if t > 20 else 1.0), 0.01, 1.0 if t % 7 else 0.5) for t in range(1, 41)]
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ca, \
            osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as cb:
        osr.adamw_graph_create(cb, b[0], b[1], b[2], b[3])
        for t, lr, wd, clip in sched:
            synth_dev.fill_grads(a[1], 7, t, 1e-2, 0.01, 100.0)
            synth_dev.fill_grads(b[1], 7, t, 1e-2, 0.01, 100.0)
            osr.adamw_clip_step(ca, a[0], a[1], a[2], a[3], t, lr, wd, clip)
            osr.adamw_graph_step(cb, t, lr, wd, clip)
            na, sa = osr.adamw_last_norm(ca)
            nb, sb = osr.adamw_last_norm(cb)
            assert (na, sa) == (nb, sb)
        for x, y in zip(a, b):
            assert torch.equal(x, y)
        osr.adamw_graph_destroy(cb)
        with pytest.raises(osr.AdamWError) as e:
            osr.adamw_graph_step(cb, 41, 1e-3, 0.0, 1.0)
        assert e.value.status == osr.ESTATE


def test_captured_steps_replay_and_leave_no_error(dev):
    """Steps captured into a torch CUDA graph replay to the same bits as
    eager steps (t fixed inside the graph), and neither the capture nor the
    context's destruction leaves a pending CUDA error behind: a new context
    can be created afterwards."""
    n = 100_003
    a = _state(dev, n)
    b = _state(dev, n)
    synth_dev.fill_grads(a[1], 7, 1, 1e-2)
    b[1].copy_(a[1])
    ctx_a = osr.adamw_create(n, flags=osr.CREATE_NO_CKPT)
    ctx_b = osr.adamw_create(n, flags=osr.CREATE_NO_CKPT)
    cap = torch.cuda.Stream()
    gr = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gr, stream=cap):
            for _ in range(3):
                osr.adamw_clip_step(ctx_b, b[0], b[1], b[2], b[3], 5, 1e-3, 0.01, 1.0, stream=cap)
    for _ in range(2):
        gr.replay()
        for _ in range(3):
            osr.adamw_clip_step(ctx_a, a[0], a[1], a[2], a[3], 5, 1e-3, 0.01, 1.0)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    del gr
    ctx_a.close()
    ctx_b.close()
    with osr.adamw_create(n) as ctx:
        assert ctx.n == n
