"""Device twin of the synthetic input generator (``gen.cu``): builds and
loads ``_gen.so`` and fills torch CUDA tensors with the same draws that
``synthetic.draw`` makes on the host, bit for bit."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

from . import device_args, STREAM_G, STREAM_W

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "gen.cu")
LIBRARY = os.path.join(HERE, "_gen.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", SOURCE, "-o", LIBRARY + ".part"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("building gen.cu failed:\n" + r.stdout + r.stderr)
    os.replace(LIBRARY + ".part", LIBRARY)
    return LIBRARY


def _library():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIBRARY)
            lib.synth_fill.restype = ctypes.c_int
            lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                       ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_float, ctypes.c_void_p]
            _lib = lib
        return _lib


def fill(out, seed: int, stream_id: int, step: int, sigma: float,
         outlier_frac: float = 0.0, outlier_mult: float = 1.0, cuda_stream=None):
    """Fills the float32 CUDA tensor ``out`` (contiguous) with a draw."""
    import torch
    assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
    a = device_args(seed, stream_id, step, sigma, outlier_frac, outlier_mult)
    s = (cuda_stream or torch.cuda.current_stream()).cuda_stream
    rc = _library().synth_fill(out.data_ptr(), out.numel(), a["key"], a["scale"],
                               a["okey"], a["othr"], a["omul"], s)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with CUDA error {rc}")
    return out


def fill_grads(out, seed, step, sigma, outlier_frac=0.0, outlier_mult=1.0, cuda_stream=None):
    return fill(out, seed, STREAM_G, step, sigma, outlier_frac, outlier_mult, cuda_stream)


def fill_weights(out, seed, sigma=0.02, cuda_stream=None):
    return fill(out, seed, STREAM_W, 0, sigma, cuda_stream=cuda_stream)
