"""GPU checkpoint runtime: asynchronous writes overlapping later steps,
rotation, the cadence policy, and SIGUSR1 / SIGTERM handled at step
boundaries by a training process whose last checkpoint resumes
bit-identically."""
import os
import signal
import subprocess
import sys

import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def gen_state(dev, n, seed=7):
    hw = synthetic.weights(seed, n=n)
    hm = synthetic.draw(seed, 11, 0, 1e-3, n=n)
    hv = np.abs(synthetic.draw(seed, 12, 0, 1e-5, n=n))
    return [torch.from_numpy(h).to(dev) for h in (hw, hm, hv)], (hw, hm, hv)


@pytest.mark.parametrize("flags", [osr.CKPT_DIRECT, 0])
def test_async_write_overlaps_steps(dev, oracle, tmp_path, flags):
    n = 3_000_001
    (w, m, v), hstate = gen_state(dev, n)
    g = torch.empty(n, device=dev)
    with osr.adamw_create(n) as ctx:
        osr.ckpt_set_options(ctx, 0, flags)
        side = torch.cuda.Stream()
        osr.ckpt_pack(ctx, 5, w, m, v, side_stream=side)
        osr.ckpt_write_async(ctx, str(tmp_path))
        for t in range(6, 12):
            synth_dev.fill_grads(g, 7, t, 1e-3)
            osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
        path = osr.ckpt_wait(ctx)
        assert osr.ckpt_wait(ctx) == path  # idempotent
    assert open(path, "rb").read() == oracle.pack(5, *hstate).tobytes()


def test_rotation_through_the_policy(dev, tmp_path):
    n = 100_000
    (w, m, v), _ = gen_state(dev, n)
    g = torch.empty(n, device=dev)
    with osr.adamw_create(n) as ctx:
        osr.ckpt_set_options(ctx, keep=2)
        actions = []
        for t in range(1, 9):
            synth_dev.fill_grads(g, 7, t, 1e-2)
            osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
            actions.append(osr.ckpt_step_end(ctx, t, w, m, v, str(tmp_path), every=2))
        last = osr.ckpt_wait(ctx)
        snap = [x.cpu().numpy() for x in (w, m, v)]
    assert actions == [0, 1, 0, 1, 0, 1, 0, 1]
    assert sorted(os.listdir(tmp_path)) == ["step_000006.bin", "step_000008.bin"]
    assert os.path.basename(last) == "step_000008.bin"
    body = np.fromfile(last, dtype="<f4", offset=8)
    assert body.tobytes() == b"".join(a.tobytes() for a in snap)


def test_write_error_is_reported(dev, tmp_path):
    n = 1000
    (w, m, v), _ = gen_state(dev, n)
    with osr.adamw_create(n) as ctx:
        osr.ckpt_pack(ctx, 1, w, m, v)
        osr.ckpt_write_async(ctx, str(tmp_path / "no_such_dir"))
        with pytest.raises(osr.AdamWError) as e:
            osr.ckpt_wait(ctx)
        assert e.value.status == osr.EIO
        osr.ckpt_write_async(ctx, str(tmp_path / "no_such_dir"))
        osr.ckpt_pack(ctx, 2, w, m, v)  # waits for the failing write
        with pytest.raises(osr.AdamWError):  # uncollected failure surfaces here
            osr.ckpt_write_async(ctx, str(tmp_path))
        osr.ckpt_write(ctx, str(tmp_path))
    assert os.listdir(tmp_path) == ["step_000002.bin"]


def uninterrupted(dev, n, steps):
    w = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, 7)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    g = torch.empty(n, device=dev)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        for t in range(1, steps + 1):
            synth_dev.fill_grads(g, 7, t, 1e-2, 0.01, 100.0)
            osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
    return w, m, v


def test_sigusr1_then_sigterm(dev, tmp_path):
    """A child training process gets SIGUSR1 (checkpoint, keeps training)
    and then SIGTERM (checkpoint after the step in flight, exits 0).  Both
    files hold exactly the uninterrupted state at their step; resuming from
    the SIGTERM file continues bit-identically."""
    n = 1_000_003
    p = subprocess.Popen([sys.executable, os.path.join(HERE, "signal_train_child.py"),
                          str(n), str(tmp_path), "100000"],
                         stdout=subprocess.PIPE, text=True)
    seen = []
    try:
        assert p.stdout.readline().strip() == "ready"
        sent_usr1 = sent_term = False
        for line in p.stdout:
            step, action = (int(x) for x in line.split()[1:])
            seen.append((step, action))
            if step >= 20 and not sent_usr1:
                p.send_signal(signal.SIGUSR1)
                sent_usr1 = True
            if step >= 60 and not sent_term:
                p.send_signal(signal.SIGTERM)
                sent_term = True
            if action == osr.CKPT_ACTION_EXIT:
                break
        assert p.wait(timeout=120) == 0
    finally:
        if p.poll() is None:
            p.kill()
            p.wait()
    written = [s for s, a in seen if a == osr.CKPT_ACTION_WRITING]
    exits = [s for s, a in seen if a == osr.CKPT_ACTION_EXIT]
    assert len(written) == 1 and len(exits) == 1 and written[0] >= 20 and exits[0] >= 60
    files = sorted(os.listdir(tmp_path))
    assert files == [f"step_{written[0]:06d}.bin", f"step_{exits[0]:06d}.bin"]
    for s in (written[0], exits[0]):
        ref = uninterrupted(dev, n, s)
        body = np.fromfile(tmp_path / f"step_{s:06d}.bin", dtype="<f4", offset=8)
        assert body.tobytes() == b"".join(x.cpu().numpy().tobytes() for x in ref)
    # resume from the SIGTERM checkpoint for 10 more steps
    s = exits[0]
    w, m, v = (torch.empty(n, device=dev) for _ in range(3))
    g = torch.empty(n, device=dev)
    with osr.adamw_create(n) as ctx:
        assert osr.ckpt_read(ctx, str(tmp_path / f"step_{s:06d}.bin"), w, m, v) == s
        for t in range(s + 1, s + 11):
            synth_dev.fill_grads(g, 7, t, 1e-2, 0.01, 100.0)
            osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
    ref = uninterrupted(dev, n, s + 10)
    for a, b in zip((w, m, v), ref):
        assert torch.equal(a, b)
