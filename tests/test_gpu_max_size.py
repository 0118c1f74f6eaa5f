"""The largest state the checkpoint header allows: n = 2^31 - 1 parameters
(an int32 count; 34.4 GB of w, g, m, v).  n is odd, so the fused kernel's
float4 pass ends with a 3-element tail.  The norm against the oracle over
all 2^31 - 1 values, and one step at sampled elements (the first and last
few, tile edges, random) against the oracle element by element."""
import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from parity import RTOL_NORM, RTOL_ONE_STEP, Running, assert_within, sample_indices

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu

N_MAX = (1 << 31) - 1
LR, WD, CLIP = 3e-3, 0.01, 1.0


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def test_one_step_at_the_largest_n(dev, oracle):
    n = N_MAX
    assert osr.ckpt_file_size(n) == 8 + 12 * n
    w = torch.empty(n, device=dev)
    g = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, 7)
    synth_dev.fill_grads(g, 7, 1, 1e-3, 0.001, 1000.0)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    idx = np.unique(np.concatenate([sample_indices(n, 100_000),
                                    np.arange(n - 16, n, dtype=np.int64)]))
    idx_t = torch.from_numpy(idx).to(dev)
    hw = w[idx_t].cpu().numpy()
    hg_s = g[idx_t].cpu().numpy()
    assert hw.tobytes() == synthetic.weights(7, idx=idx).tobytes()
    onorm = oracle.global_norm(g.cpu().numpy())
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_clip_step(ctx, w, g, m, v, 1, LR, WD, CLIP)
        norm, scale = osr.adamw_last_norm(ctx)
    assert abs(norm - onorm) <= RTOL_NORM * onorm, (norm, onorm)
    s = oracle.clip_scale(onorm, CLIP)
    sub = np.arange(idx.size)
    z = np.zeros(idx.size, np.float32)
    want = oracle.adamw_at(sub, hw, hg_s, z, z, s, 1, LR, WD)
    terms = oracle.adamw_terms_at(sub, hw, hg_s, z, z, s, 1, LR, WD)
    got = [x[idx_t].cpu().numpy() for x in (w, m, v)]
    assert_within(got, want, Running().update(terms, LR, WD, 1), RTOL_ONE_STEP, "n = 2^31 - 1")
    del w, g, m, v
    torch.cuda.empty_cache()


def test_largest_n_is_accepted_and_one_more_refused(dev):
    with osr.adamw_create(N_MAX, flags=osr.CREATE_NO_CKPT) as ctx:
        assert ctx.n == N_MAX
    with pytest.raises(osr.AdamWError) as e:
        osr.adamw_create(N_MAX + 1, flags=osr.CREATE_NO_CKPT)
    assert e.value.status == osr.EINVAL
