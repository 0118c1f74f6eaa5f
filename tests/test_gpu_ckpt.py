"""GPU checkpoint path: the packed image and the written file equal the
oracle's image of the same state byte for byte; reading restores the state
bit for bit and refuses bad files without touching device memory; resuming
from the file continues bit-identically to an uninterrupted run."""
import os

import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from synthetic import workloads as W

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def state(dev, n, seed=7):
    """(device tensors, host arrays) of a generator-made w, m, v."""
    hw = synthetic.weights(seed, n=n)
    hm = synthetic.draw(seed, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(seed, 12, 0, 1e-5, n=n))
    return [torch.from_numpy(h).to(dev) for h in (hw, hm, hv)], (hw, hm, hv)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9, 1001, 65536, 65536 + 2,
                               1_000_001, 1_000_003, (1 << 24) + 3])
@pytest.mark.parametrize("copy", ["kernel", "copy_engine"])
def test_pack_write_bytes_match_oracle(dev, oracle, tmp_path, n, copy):
    """Both ways from the staging to the pinned image (the side-stream
    kernel -- each region copied as 0-3 head floats up to a 16-byte boundary,
    aligned 16-byte units assembled from two staging float4, a tail; n % 4
    covers every head length, n <= 9 the cases with no or one unit -- and the
    copy engine) give the oracle's bytes."""
    (w, m, v), hstate = state(dev, n)
    with osr.adamw_create(n) as ctx:
        osr.ckpt_set_options(ctx, 0, osr.CKPT_DIRECT | (osr.CKPT_COPY_ENGINE
                                                         if copy == "copy_engine" else 0))
        side = torch.cuda.Stream()
        osr.ckpt_pack(ctx, 80, w, m, v, side_stream=side)
        path = osr.ckpt_write(ctx, str(tmp_path))
    assert os.path.basename(path) == "step_000080.bin"
    data = open(path, "rb").read()
    assert len(data) == 8 + 12 * n == osr.ckpt_file_size(n)
    want = oracle.pack(80, *hstate)
    assert data == want.tobytes()
    assert not os.path.exists(path + ".tmp")
    st, step, ow, om, ov = oracle.ckpt_read(path, n)
    assert st == 0 and step == 80


def test_read_restores_bit_exact(dev, oracle, tmp_path):
    n = 100_003
    hw, hm, hv = (np.random.default_rng(i).standard_normal(n).astype(np.float32)
                  for i in range(3))
    path = oracle.ckpt_write(str(tmp_path), 4585, hw, hm, hv)
    w, m, v = (torch.full((n,), 7.0, device=dev) for _ in range(3))
    with osr.adamw_create(n) as ctx:
        assert osr.ckpt_read(ctx, path, w, m, v) == 4585
    for t, h in ((w, hw), (m, hm), (v, hv)):
        assert t.cpu().numpy().tobytes() == h.tobytes()


def test_read_refuses_bad_files_and_leaves_state(dev, oracle, tmp_path):
    n = 4096
    z = np.zeros(n, np.float32)
    good = oracle.ckpt_write(str(tmp_path), 3, z + 1, z + 2, z + 3)
    data = open(good, "rb").read()
    w, m, v = (torch.full((n,), 9.0, device=dev) for _ in range(3))
    cases = {"trunc.bin": (data[:-1], osr.ESIZE),
             "long.bin": (data + b"xx", osr.ESIZE),
             "hdr.bin": (data[:6], osr.ESIZE)}
    with osr.adamw_create(n) as ctx:
        for name, (payload, status) in cases.items():
            p = tmp_path / name
            p.write_bytes(payload)
            with pytest.raises(osr.AdamWError) as e:
                osr.ckpt_read(ctx, str(p), w, m, v)
            assert e.value.status == status
        other = oracle.ckpt_write(str(tmp_path / ".."), 3, np.zeros(n + 4, np.float32),
                                  np.zeros(n + 4, np.float32), np.zeros(n + 4, np.float32))
        with pytest.raises(osr.AdamWError) as e:
            osr.ckpt_read(ctx, other, w, m, v)
        assert e.value.status == osr.EMISMATCH
        os.unlink(other)
    for t in (w, m, v):
        assert bool((t == 9.0).all())


def test_pack_overlaps_next_step(dev, oracle, tmp_path):
    """The pack snapshots the state at the step boundary: steps launched
    right after it (before the side-stream copy finishes) do not leak into
    the file."""
    n = 4_000_000
    (w, m, v), hstate = state(dev, n)
    g = torch.empty(n, device=dev)
    with osr.adamw_create(n) as ctx:
        side = torch.cuda.Stream()
        osr.ckpt_pack(ctx, 1, w, m, v, side_stream=side)
        for t in range(2, 6):
            synth_dev.fill_grads(g, 7, t, 1e-3)
            osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
        path = osr.ckpt_write(ctx, str(tmp_path))
        assert not torch.equal(w.cpu(), torch.from_numpy(hstate[0]))
    assert open(path, "rb").read() == oracle.pack(1, *hstate).tobytes()


def run_steps(ctx, w, g, m, v, wl, t0, t1, outliers=True):
    for t in range(t0, t1 + 1):
        if outliers:
            synth_dev.fill_grads(g, wl.seed, t, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
        else:
            synth_dev.fill_grads(g, wl.seed, t, wl.grad_sigma)
        osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)


def resume_case(dev, tmp_path, wl, total, at, table=None):
    n = wl.n
    off, num = table if table else (None, None)
    g = torch.empty(n, device=dev)
    w = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    w0 = w.clone()
    with osr.adamw_create(n, off, num) as ctx:
        run_steps(ctx, w, g, m, v, wl, 1, total)
        ref = [t.clone() for t in (w, m, v)]
        # interrupted run: `at` steps, checkpoint, fresh buffers, read, rest
        w.copy_(w0)
        m.zero_()
        v.zero_()
        run_steps(ctx, w, g, m, v, wl, 1, at)
        osr.ckpt_pack(ctx, at, w, m, v, side_stream=torch.cuda.Stream())
        path = osr.ckpt_write(ctx, str(tmp_path))
        assert os.path.getsize(path) == 8 + 12 * n
        w.fill_(float("nan"))
        m.fill_(float("nan"))
        v.fill_(float("nan"))
    with osr.adamw_create(n, off, num) as ctx2:  # as after a process restart
        step = osr.ckpt_read(ctx2, path, w, m, v)
        assert step == at
        run_steps(ctx2, w, g, m, v, wl, step + 1, total)
    for a, b in zip((w, m, v), ref):
        assert torch.equal(a, b)
    return path


def test_resume_flat_65536_80_steps(dev, tmp_path):
    wl = W.flat_65k()
    resume_case(dev, tmp_path, wl, 80, 40)


def test_resume_gpt_110m_200_steps(dev, tmp_path):
    """Configuration gpt-110M-resume: 200 steps with a checkpoint at 100,
    reloaded from the file into a fresh context, bit-identical at 200."""
    wl = W.gpt_110m_resume()
    resume_case(dev, tmp_path, wl, 200, 100, table=wl.table())
    torch.cuda.empty_cache()
