"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every function include/*.h declares, validates offset tables before touching
CUDA, and its checkpoint writer/prober agree byte for byte with the oracle's."""
import glob
import os
import re
import signal
import struct
import subprocess
import sys
import time

import numpy as np
import pytest

import optimizer_step_resumable_gb300 as osr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"ADAMW_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("adamw_create", "adamw_destroy", "grad_global_norm", "adamw_clip_step",
                 "ckpt_pack", "ckpt_write", "ckpt_read"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", osr.LIBRARY],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(declared_functions()) <= exported
    # nothing but the C ABI leaks out (kernels and helpers are hidden)
    assert not [s for s in exported if s.startswith("_ZN3osr")]


def test_binding_covers_the_abi():
    assert sorted(osr.SIGNATURES) == declared_functions()


def test_strerror(lib):
    assert osr.adamw_strerror(osr.OK) == "ADAMW_OK"
    assert "finite" in osr.adamw_strerror(osr.ENONFINITE)
    assert osr.adamw_strerror(12345) == "unknown status"


def test_file_size(lib):
    assert osr.ckpt_file_size(12_800_000) == 153_600_008
    assert osr.ckpt_file_size(110_418_432) == 1_325_021_192
    assert osr.ckpt_file_size(1 << 30) == 12_884_901_896
    assert osr.ckpt_file_size(-1) == -1 and osr.ckpt_file_size(1 << 31) == -1


@pytest.mark.parametrize("case", [
    dict(n=0, off=None, num=None),
    dict(n=1 << 31, off=None, num=None),
    dict(n=10, off=[0, 5], num=[5, 4]),        # short of n
    dict(n=10, off=[0, 4], num=[5, 5]),        # overlap
    dict(n=10, off=[0, 6], num=[5, 4]),        # gap
    dict(n=10, off=[5, 0], num=[5, 5]),        # unsorted
    dict(n=10, off=[0, 5, 10], num=[5, 5, 0]),  # empty tensor
    dict(n=10, off=[0], num=[11]),             # past the end
])
def test_create_rejects_bad_tables_before_cuda(lib, case):
    with pytest.raises(osr.AdamWError) as e:
        osr.adamw_create(case["n"], case["off"], case["num"])
    assert e.value.status == osr.EINVAL


def test_create_without_gpu_fails_cleanly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(osr.AdamWError) as e:
        osr.adamw_create(1000)
    assert e.value.status == osr.ECUDA


def _state(n, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(n).astype(np.float32) for _ in range(3)]


@pytest.mark.parametrize("n", [1, 5, 1000])
def test_host_writer_matches_oracle_bytes(lib, oracle, tmp_path, n):
    w, m, v = _state(n, n)
    (tmp_path / "a").mkdir()
    (tmp_path / "b").mkdir()
    p1 = osr.ckpt_write_host(str(tmp_path / "a"), 100, w, m, v)
    p2 = oracle.ckpt_write(str(tmp_path / "b"), 100, w, m, v)
    assert os.path.basename(p1) == os.path.basename(p2) == "step_000100.bin"
    assert open(p1, "rb").read() == open(p2, "rb").read() == oracle.pack(100, w, m, v).tobytes()
    assert not os.path.exists(p1 + ".tmp")
    assert osr.ckpt_probe(p1, n) == (100, n)
    assert osr.ckpt_probe(p2) == (100, n)


def test_probe_rejects_bad_files(lib, oracle, tmp_path):
    n = 16
    w, m, v = _state(n, 1)
    good = oracle.ckpt_write(str(tmp_path), 7, w, m, v)
    data = open(good, "rb").read()
    cases = {
        "trunc": (data[:-4], osr.ESIZE), "extra": (data + b"\0", osr.ESIZE),
        "short": (data[:5], osr.ESIZE), "empty": (b"", osr.ESIZE),
        "other_n": (struct.pack("<ii", 7, n + 1) + data[8:], osr.EMISMATCH),
        "neg_n": (struct.pack("<ii", 7, -1) + data[8:], osr.EFORMAT),
        "neg_step": (struct.pack("<ii", -2, n) + data[8:], osr.EFORMAT),
    }
    for name, (payload, status) in cases.items():
        p = tmp_path / (name + ".bin")
        p.write_bytes(payload)
        with pytest.raises(osr.AdamWError) as e:
            osr.ckpt_probe(str(p), n)
        assert e.value.status == status, name
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_probe(str(tmp_path / "absent.bin"), n)
    assert e.value.status == osr.EIO
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_write_host(str(tmp_path / "no_such_dir"), 1, w, m, v)
    assert e.value.status == osr.EIO


CHILD = r"""
import sys, numpy as np
sys.path.insert(0, {root!r})
import optimizer_step_resumable_gb300 as osr
n = {n}
a = [np.full(n, 1.0, np.float32), np.full(n, 2.0, np.float32), np.full(n, 3.0, np.float32)]
b = [np.full(n, -1.0, np.float32), np.full(n, -2.0, np.float32), np.full(n, -3.0, np.float32)]
osr.ckpt_write_host({d!r}, 100, *a)
print("ready", flush=True)
while True:
    osr.ckpt_write_host({d!r}, 100, *b)
    osr.ckpt_write_host({d!r}, 100, *a)
"""


def test_killed_writer_leaves_a_complete_file(lib, oracle, tmp_path):
    """SIGKILL the writer at random points while it rewrites the same
    checkpoint: the final name always holds one complete image (the old or
    the new one), never a partial one; a stray .tmp is ignored."""
    n = 1 << 21
    na = [np.full(n, x, np.float32) for x in (1.0, 2.0, 3.0)]
    nb = [np.full(n, -x, np.float32) for x in (1.0, 2.0, 3.0)]
    images = {oracle.pack(100, *na).tobytes(), oracle.pack(100, *nb).tobytes()}
    rng = np.random.default_rng(0)
    for trial in range(4):
        d = tmp_path / f"t{trial}"
        d.mkdir()
        p = subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT, n=n, d=str(d))],
                             stdout=subprocess.PIPE, text=True)
        try:
            assert p.stdout.readline().strip() == "ready"
            time.sleep(float(rng.uniform(0.01, 0.3)))
        finally:
            p.send_signal(signal.SIGKILL)
            p.wait()
        final = d / "step_000100.bin"
        assert osr.ckpt_probe(str(final), n) == (100, n)
        assert final.read_bytes() in images


def test_binding_refuses_tensors_of_another_device():
    """Pointers handed to a context must live on its device (a tensor of
    another GPU would give the kernels an address of the wrong memory)."""
    import types
    ctx = types.SimpleNamespace(device=0)
    on = lambda i: types.SimpleNamespace(get_device=lambda: i)  # noqa: E731
    osr._same_device(on(0), "w", ctx)
    osr._same_device(on(1), "w", None)  # no context: nothing to compare
    with pytest.raises(ValueError, match="cuda:1, the context on cuda:0"):
        osr._same_device(on(1), "w", ctx)
