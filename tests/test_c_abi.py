"""The C ABI from plain C: tests/c_abi/step_ckpt.c includes only
adamw_ckpt.h and the CUDA runtime, links the library, runs clipped-AdamW steps
and writes a checkpoint.  On the CPU it must compile and link as C11; on the
GPU its one-step state matches the oracle and its three-step checkpoint is
the same file, byte for byte, as the same run through the Python binding."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import synthetic
from parity import RTOL_ONE_STEP, assert_state_close

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "step_ckpt.c")
PKG = os.path.join(ROOT, "optimizer_step_resumable_gb300")
LR, WD, CLIP = 3e-3, 0.01, 1.0


def cuda_home():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return home if os.path.isdir(os.path.join(home, "include")) else None


def build_c_caller(out_dir):
    cc = shutil.which("gcc") or shutil.which("cc")
    home = cuda_home()
    if not cc or not home:
        pytest.skip("needs a C compiler and the CUDA toolkit")
    exe = os.path.join(str(out_dir), "step_ckpt")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(home, "include"), SRC, "-o", exe, "-L", PKG, "-loptstep",
           "-L", os.path.join(home, "lib64"), "-lcudart", "-Wl,-rpath," + PKG]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_caller_compiles_and_links_as_c11(lib, tmp_path):
    assert os.access(build_c_caller(tmp_path), os.X_OK)


def run_c(exe, tmp_path, n, w, g, steps, tag):
    wf, gf = tmp_path / f"w_{tag}.f32", tmp_path / f"g_{tag}.f32"
    w.tofile(wf)
    g.tofile(gf)
    out = tmp_path / f"ckpt_{tag}"
    out.mkdir()
    r = subprocess.run([exe, str(n), str(wf), str(gf), str(steps), repr(LR), repr(WD),
                        repr(CLIP), str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    path, norm, scale = r.stdout.split()
    return path, float(norm), float(scale)


@pytest.mark.gpu
def test_c_caller_matches_oracle_and_python_binding(lib, oracle, tmp_path):
    torch = pytest.importorskip("torch")
    import optimizer_step_resumable_gb300 as osr
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    exe = build_c_caller(tmp_path)
    n = 100_003  # several tiles and a ragged tail: the two-launch step
    w0 = synthetic.weights(7, n=n)
    g = synthetic.grads(7, 1, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
    zeros = np.zeros(n, np.float32)

    # one step from plain C against the oracle
    path, norm, _ = run_c(exe, tmp_path, n, w0, g, 1, "one")
    st, step, cw, cm, cv = oracle.ckpt_read(path, n)
    assert st == 0 and step == 1
    onorm = oracle.global_norm(g)
    assert abs(norm - onorm) <= 1e-6 * onorm
    s = oracle.clip_scale(onorm, CLIP)
    idx = np.arange(n)
    want = oracle.adamw_at(idx, w0, g, zeros, zeros, s, 1, LR, WD)
    terms = oracle.adamw_terms_at(idx, w0, g, zeros, zeros, s, 1, LR, WD)
    assert_state_close((cw, cm, cv), want, terms, RTOL_ONE_STEP, "C caller", lr=LR, t=1)

    # three steps from plain C and through the Python binding: the same file
    path_c, norm_c, scale_c = run_c(exe, tmp_path, n, w0, g, 3, "three")
    dev = torch.device("cuda:0")
    w, gd = torch.from_numpy(w0).to(dev), torch.from_numpy(g).to(dev)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    out = tmp_path / "ckpt_py"
    out.mkdir()
    with osr.adamw_create(n) as ctx:
        for t in (1, 2, 3):
            osr.adamw_clip_step(ctx, w, gd, m, v, t, LR, WD, CLIP)
        norm_p, scale_p = osr.adamw_last_norm(ctx)
        osr.ckpt_pack(ctx, 3, w, m, v)
        path_p = osr.ckpt_write(ctx, str(out))
    assert open(path_c, "rb").read() == open(path_p, "rb").read()
    assert norm_c == norm_p and np.float32(scale_c) == np.float32(scale_p)
