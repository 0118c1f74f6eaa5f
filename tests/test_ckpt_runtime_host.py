"""Host side of the checkpoint runtime (no GPU): the image writer with and
without O_DIRECT, rotation, and the SIGTERM / SIGUSR1 request flags."""
import os
import signal
import subprocess
import sys
import time

import numpy as np
import pytest

import optimizer_step_resumable_gb300 as osr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def aligned_image(oracle, step, n, pad_to=4096, offset=0):
    rng = np.random.default_rng(n)
    w, m, v = (rng.standard_normal(n).astype(np.float32) for _ in range(3))
    img = oracle.pack(step, w, m, v)
    cap = (img.size + pad_to - 1) // pad_to * pad_to
    raw = np.full(cap + 2 * pad_to, 0xAB, np.uint8)
    start = (-raw.ctypes.data) % pad_to + offset
    buf = raw[start:start + cap]
    buf[:img.size] = img
    return img, buf


@pytest.mark.parametrize("n", [1, 1000, 341_333])
@pytest.mark.parametrize("flags", [osr.CKPT_DIRECT, 0])
def test_image_writer_bytes(lib, oracle, tmp_path, n, flags):
    img, buf = aligned_image(oracle, 42, n)
    assert buf.ctypes.data % 4096 == 0
    path = osr.ckpt_write_image(str(tmp_path), buf, img.size, flags)
    assert os.path.basename(path) == "step_000042.bin"
    assert open(path, "rb").read() == img.tobytes()  # padding cut off
    assert not os.path.exists(path + ".tmp")


def test_image_writer_unaligned_falls_back(lib, oracle, tmp_path):
    img, buf = aligned_image(oracle, 7, 999, offset=8)
    assert buf.ctypes.data % 4096 == 8
    path = osr.ckpt_write_image(str(tmp_path), buf, img.size, osr.CKPT_DIRECT)
    assert open(path, "rb").read() == img.tobytes()


def test_image_writer_rejects_inconsistent_header(lib, oracle, tmp_path):
    img, buf = aligned_image(oracle, 7, 100)
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_write_image(str(tmp_path), buf, img.size - 4)
    assert e.value.status == osr.EINVAL


def test_rotation_keeps_the_newest(lib, tmp_path):
    z = np.zeros(8, np.float32)
    for s in (1, 2, 3, 10, 1000000, 99):
        osr.ckpt_write_host(str(tmp_path), s, z, z, z)
    others = ["step_abc.bin", "step_000002.bin.tmp", "other.bin", "step_1.bin.bak", "step_.bin"]
    for nm in others:
        (tmp_path / nm).write_bytes(b"x")
    assert osr.ckpt_rotate(str(tmp_path), 0) == 0
    assert osr.ckpt_rotate(str(tmp_path), 3) == 3
    left = sorted(os.listdir(tmp_path))
    assert left == sorted(others + ["step_000099.bin", "step_1000000.bin", "step_000010.bin"])
    assert osr.ckpt_rotate(str(tmp_path), 3) == 0
    with pytest.raises(osr.AdamWError):
        osr.ckpt_rotate(str(tmp_path / "missing"), 2)


CHILD = r"""
import sys, time
sys.path.insert(0, {root!r})
import optimizer_step_resumable_gb300 as osr
osr.ckpt_signals_install(osr.CKPT_REQ_WRITE | osr.CKPT_REQ_EXIT)
print("ready", flush=True)
deadline = time.time() + 60
while time.time() < deadline:
    req = osr.ckpt_signals_take()
    if req & osr.CKPT_REQ_EXIT:
        print("exit", flush=True)
        sys.exit(0)
    if req & osr.CKPT_REQ_WRITE:
        print("write", flush=True)
    time.sleep(0.005)
sys.exit(3)
"""


def test_signals_become_requests(lib):
    """SIGUSR1 -> a write request, the process keeps running; SIGTERM -> an
    exit request the loop acts on (the default action is replaced)."""
    p = subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)],
                         stdout=subprocess.PIPE, text=True)
    try:
        assert p.stdout.readline().strip() == "ready"
        for _ in range(2):
            p.send_signal(signal.SIGUSR1)
            assert p.stdout.readline().strip() == "write"
        p.send_signal(signal.SIGTERM)
        assert p.stdout.readline().strip() == "exit"
        assert p.wait(timeout=30) == 0
    finally:
        if p.poll() is None:
            p.kill()
            p.wait()


def test_signal_mask_validation(lib):
    with pytest.raises(osr.AdamWError):
        osr.ckpt_signals_install(4)
    assert osr.ckpt_signals_take() == 0
