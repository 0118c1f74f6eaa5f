"""Every kernel stays inside the caller's arrays.  Each array is a view into
a larger buffer whose guard regions before and after are filled with a
sentinel bit pattern; after steps through every path at sizes around every
edge (tiles, chunks, float4 tails, the one-launch limit), the guards must be
bit-unchanged.  Aligned views take the vector kernels, views one element off
take the scalar ones."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

GUARD = 1024           # elements of guard on each side
SENTINEL = 0x7FC0DEAD  # a NaN pattern no kernel writes


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


class Guarded:
    def __init__(self, dev, n, dtype=torch.float32, offset=0, fill=0.0):
        self.n, self.off = n, GUARD + offset
        self.buf = torch.empty(n + 2 * GUARD + offset, dtype=dtype, device=dev)
        if dtype == torch.float32:
            self.buf.view(torch.int32).fill_(SENTINEL)
        else:
            self.buf.view(torch.int16).fill_(0x7E5A)
        self.view = self.buf[self.off:self.off + n]
        self.view.fill_(fill)
        self.before = self.raw()

    def raw(self):
        ints = torch.int16 if self.buf.element_size() == 2 else torch.int32
        return self.buf.view(ints).cpu().numpy().tobytes()

    def check(self):
        now = self.raw()
        es = self.buf.element_size()
        lo, hi = self.off * es, (self.off + self.n) * es
        assert now[:lo] == self.before[:lo], "write before the array"
        assert now[hi:] == self.before[hi:], "write past the array"


# (from 2^24 the fused and pack kernels hand chunks out by their counters)
SIZES = [1, 2, 3, 4, 5, 7, 8, 9, 31, 33, 1023, 1025, 2047, 2049, 8191, 8193,
         65537, (1 << 19) - 1, (1 << 19) + 3, 3 * 8192 * 608 + 5, (1 << 24) + 2, (1 << 24) + 5]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("offset", [0, 1])
def test_step_paths_stay_in_bounds(dev, n, offset):
    w = Guarded(dev, n, offset=offset, fill=0.5)
    g = Guarded(dev, n, offset=offset, fill=1e-3)
    m = Guarded(dev, n, offset=offset)
    v = Guarded(dev, n, offset=offset)
    k = max(1, n // 3)
    off, num = [0, k], [k, n - k]
    table = (off, num) if n - k > 0 else (None, None)
    with osr.adamw_create(n, *table) as ctx:
        if table[0] is not None:
            osr.adamw_set_decay_mask(ctx, [0, 1])
        for t, flags in ((1, 0), (2, osr.LAUNCH_NO_ONEPASS), (3, 0)):
            osr.adamw_set_launch_options(ctx, flags)
            osr.adamw_clip_step_ex(ctx, w.view, g.view, m.view, v.view, t, 1e-3, 0.01, 1.0,
                                   zero_grad=(t == 3))
            osr.adamw_last_norm(ctx)
        osr.ckpt_pack(ctx, 3, w.view, m.view, v.view)
        osr.ckpt_wait(ctx)
        torch.cuda.synchronize()
    for a in (w, g, m, v):
        a.check()


@pytest.mark.parametrize("n", [1, 3, 4, 5, 9, 2049, 8193, 65537, (1 << 19) + 3,
                               (1 << 24) + 3])
def test_mixed_paths_stay_in_bounds(dev, n):
    w = Guarded(dev, n, fill=0.5)
    m = Guarded(dev, n)
    v = Guarded(dev, n)
    g = Guarded(dev, n, dtype=torch.bfloat16, fill=1e-3)
    lp = Guarded(dev, n, dtype=torch.bfloat16)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step_mixed(ctx, w.view, g.view, m.view, v.view, 1, 1e-3, 0.01, 1.0,
                                  w_lp=lp.view, zero_grad=True)
        osr.adamw_last_norm(ctx)
        torch.cuda.synchronize()
    for a in (w, g, m, v, lp):
        a.check()
