"""The allocation-free step, for callers that must not allocate GPU memory.

Some callers cannot create a context, because adamw_create allocates: code
that runs inside a framework or server owning all device memory through its
own pool, plug-ins given only their input and output buffers, and
latency-critical paths where cudaMalloc would synchronise the device.  They
call adamw_clip_step_noalloc, whose scratch is a fixed static device array.
These checks call it through the C ABI and compare it with the context-based
adamw_clip_step on two calls in a row, with the parity tolerance of the other
tests.  This file is collected last; it passes alone in a fresh process and
after the other tests (the shared array keeps the last call's contents, and
each call clears what must start at zero)."""
import numpy as np
import pytest

import synthetic
from parity import FLOOR, RTOL_NORM, RTOL_ONE_STEP

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _close(a, b, rtol):
    a = a.cpu().numpy().astype(np.float64)
    b = b.cpu().numpy().astype(np.float64)
    bound = rtol * np.maximum(np.abs(a), np.abs(b)) + FLOOR
    return bool(np.all(np.abs(a - b) <= bound))


@pytest.mark.parametrize("n", [65536 + 37, 1_000_003, (1 << 24) + 5])
def test_noalloc_step_matches_context_step(dev, n):
    """(2^24 + 5: the context step hands chunks out by its counter, the
    no-alloc step keeps the fixed assignment.)"""
    w0 = torch.from_numpy(synthetic.weights(7, n=n)).to(dev)
    states = [[w0.clone(), torch.zeros(n, device=dev), torch.zeros(n, device=dev)]
              for _ in range(2)]
    norm_out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    lr, wd, clip = 3e-3, 0.01, 1.0
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in (1, 2):  # two calls in a row
            g = torch.from_numpy(synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01,
                                                 outlier_mult=100.0)).to(dev)
            w, m, v = states[0]
            osr.adamw_clip_step(ctx, w, g, m, v, t, lr, wd, clip)
            ref_norm, _ = osr.adamw_last_norm(ctx)
            w, m, v = states[1]
            osr.adamw_clip_step_noalloc(w, g, m, v, t, lr, wd, clip, norm_out=norm_out)
            torch.cuda.synchronize()
            got_norm = float(norm_out.item())
            assert abs(got_norm - ref_norm) <= RTOL_NORM * ref_norm, (t, got_norm, ref_norm)
            for a, b in zip(states[0], states[1]):
                assert _close(a, b, RTOL_ONE_STEP), t


def test_noalloc_rejects_sizes_beyond_its_limit(dev):
    lib = osr.library()
    x = torch.zeros(4, device=dev)
    p = x.data_ptr()
    for n in (0, -5, 1 << 31):
        st = lib.adamw_clip_step_noalloc(p, p, p, p, n, 1, 1e-3, 0.0, 1.0, 0.9, 0.999, 1e-8,
                                         None, torch.cuda.current_stream().cuda_stream)
        assert st == osr.EINVAL
        assert "2^31-1" in osr.adamw_last_error()
