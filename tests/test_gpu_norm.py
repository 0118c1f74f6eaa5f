"""GPU parity of the global gradient norm against the oracle, plus
determinism, alignment independence and edge values.  Calls go through the
C ABI (ctypes binding of liboptstep.so)."""
import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from parity import RTOL_NORM

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def gpu_norm(g_t):
    with osr.adamw_create(g_t.numel(), flags=osr.CREATE_NO_CKPT) as ctx:
        return osr.grad_global_norm(ctx, g_t)


def test_generator_device_twin_is_bit_exact(dev):
    n = 3 * 65536 + 37
    for stream, step, sigma, frac, mult in ((synthetic.STREAM_G, 1, 1e-2, 0.01, 100.0),
                                            (synthetic.STREAM_G, 77, 1e-3, 0.001, 1000.0),
                                            (synthetic.STREAM_W, 0, 0.02, 0.0, 1.0)):
        t = torch.empty(n, device=dev)
        synth_dev.fill(t, 7, stream, step, sigma, frac, mult)
        h = synthetic.draw(7, stream, step, sigma, n=n, outlier_frac=frac, outlier_mult=mult)
        assert t.cpu().numpy().tobytes() == h.tobytes()


SIZES = [1, 3, 4, 5, 1000, 8191, 8192, 8193, 65536, 65536 + 37,
         8192 * 1216 - 3, 8192 * 1216 * 3 + 4099, 12_800_000]


@pytest.mark.parametrize("n", SIZES)
def test_norm_matches_oracle(dev, oracle, n):
    g = torch.empty(n, device=dev)
    synth_dev.fill_grads(g, 7, 1, 1e-3, 0.001, 1000.0)
    want = oracle.global_norm(g.cpu().numpy())
    got = gpu_norm(g)
    assert abs(got - want) <= RTOL_NORM * want, (n, got, want, abs(got - want) / want)


def test_norm_110m_and_1b(dev, oracle):
    for n in (110_418_432, 1 << 30):
        g = torch.empty(n, device=dev)
        synth_dev.fill_grads(g, 7, 1, 1e-3, 0.001, 1000.0)
        want = oracle.global_norm(g.cpu().numpy())
        got = gpu_norm(g)
        assert abs(got - want) <= RTOL_NORM * want, (n, got, want)
        del g
        torch.cuda.empty_cache()


def test_norm_is_bit_stable(dev):
    n = 12_800_000
    g = torch.empty(n, device=dev)
    synth_dev.fill_grads(g, 7, 3, 1e-3)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        vals = {osr.grad_global_norm(ctx, g) for _ in range(10)}
    assert len(vals) == 1


def test_norm_independent_of_alignment(dev, oracle):
    """A view starting 4 bytes into a buffer takes the scalar path; the
    element-to-thread mapping is the same, so the bits are too."""
    n = 8192 * 5 + 3
    buf = torch.empty(n + 1, device=dev)
    synth_dev.fill_grads(buf, 7, 5, 1e-2, 0.01, 100.0)
    view = buf[1:]
    assert view.data_ptr() % 16 == 4
    aligned = view.clone()
    a, b = gpu_norm(view), gpu_norm(aligned)
    assert a == b
    want = oracle.global_norm(aligned.cpu().numpy())
    assert abs(a - want) <= RTOL_NORM * want


@pytest.mark.parametrize("kind", ["zeros", "huge", "tiny", "mixed", "one_big"])
def test_norm_edge_values(dev, oracle, kind):
    """Squares that overflow or underflow float32 take the exact double path."""
    n = 50_000
    rng = np.random.default_rng(11)
    if kind == "zeros":
        h = np.zeros(n, np.float32)
    elif kind == "huge":
        h = (rng.standard_normal(n) * 3e20).astype(np.float32)
    elif kind == "tiny":
        h = (rng.standard_normal(n) * 1e-25).astype(np.float32)
    elif kind == "mixed":
        h = (rng.standard_normal(n) * 10.0 ** rng.integers(-30, 30, n)).astype(np.float32)
    else:
        h = np.zeros(n, np.float32)
        h[12345] = -2.5e30
    got = gpu_norm(torch.from_numpy(h).to(dev))
    want = oracle.global_norm(h)
    assert abs(got - want) <= RTOL_NORM * want, (kind, got, want)


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_norm_nonfinite(dev, bad):
    h = np.ones(10_000, np.float32)
    h[777] = bad
    with osr.adamw_create(h.size, flags=osr.CREATE_NO_CKPT) as ctx:
        with pytest.raises(osr.NonFiniteGradient):
            osr.grad_global_norm(ctx, torch.from_numpy(h).to(dev))
        # the context stays usable
        assert osr.grad_global_norm(ctx, torch.ones(10_000, device=dev)) == 100.0


def test_norm_special_values(dev):
    for vec, want in (([3.0, 4.0], 5.0), ([0.5] * 4096, 32.0), ([0.0] * 7, 0.0)):
        assert gpu_norm(torch.tensor(vec, device=dev)) == want
