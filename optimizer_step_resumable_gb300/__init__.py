"""GB300-native clipped-AdamW optimizer step and step_NNNNNN.bin checkpoint.

Thin Python binding of the C ABI in ``include/adamw_ckpt.h`` (library
``liboptstep.so``, built in-tree by ``build.py``).  Functions carry the C
names; this module only marshals arguments: torch tensors become device
pointers, torch streams become ``cudaStream_t`` handles, non-zero statuses
become exceptions.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback, and using any function without the
built library raises ``LibraryNotBuilt``.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "liboptstep.so")

OK = 0
EINVAL, ECUDA, EIO, EFORMAT, ESIZE, EMISMATCH, ENONFINITE, ESTATE = range(-1, -9, -1)
CREATE_NO_CKPT = 1
CKPT_DIRECT = 1
CKPT_COPY_ENGINE = 2
DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2
ZERO_GRAD = 1
TENSOR_NORMS = 2
LAUNCH_NO_PDL = 1
LAUNCH_NO_ONEPASS = 2
LAUNCH_TEST_BARRIER_TIMEOUT = 4
LAUNCH_STATIC_CHUNKS = 8
CKPT_REQ_WRITE, CKPT_REQ_EXIT = 1, 2
CKPT_ACTION_NONE, CKPT_ACTION_WRITING, CKPT_ACTION_EXIT = 0, 1, 2

# ABI: name -> (restype, argtypes)
_c = ctypes
_vp = _c.c_void_p
SIGNATURES = {
    "adamw_create": (_c.c_int, [_c.c_int64, _vp, _vp, _c.c_int32, _c.c_int32,
                                _c.POINTER(_vp)]),
    "adamw_destroy": (_c.c_int, [_vp]),
    "adamw_set_hparams": (_c.c_int, [_vp, _c.c_double, _c.c_double, _c.c_double]),
    "adamw_num_params": (_c.c_int64, [_vp]),
    "adamw_num_tensors": (_c.c_int32, [_vp]),
    "grad_global_norm": (_c.c_int, [_vp, _vp, _c.POINTER(_c.c_double), _vp]),
    "adamw_clip_step": (_c.c_int, [_vp, _vp, _vp, _vp, _vp, _c.c_int32, _c.c_double,
                                   _c.c_double, _c.c_double, _vp]),
    "adamw_last_norm": (_c.c_int, [_vp, _c.POINTER(_c.c_double), _c.POINTER(_c.c_float)]),
    "adamw_clip_step_ex": (_c.c_int, [_vp, _vp, _vp, _vp, _vp, _c.c_int32, _c.c_double,
                                      _c.c_double, _c.c_double, _c.c_double, _c.c_double,
                                      _c.c_int32, _vp]),
    "grad_sumsq": (_c.c_int, [_vp, _vp, _c.POINTER(_c.c_double), _vp]),
    "grad_tensor_sumsq": (_c.c_int, [_vp, _vp, _vp, _vp]),
    "adamw_clip_step_mixed": (_c.c_int, [_vp, _vp, _vp, _c.c_int32, _vp, _vp, _vp, _c.c_int32,
                                         _c.c_int32, _c.c_double, _c.c_double, _c.c_double,
                                         _c.c_double, _c.c_double, _c.c_int32, _vp]),
    "grad_sumsq_typed": (_c.c_int, [_vp, _vp, _c.c_int32, _c.POINTER(_c.c_double), _vp]),
    "grad_sumsq_to": (_c.c_int, [_vp, _vp, _c.c_int32, _vp, _vp]),
    "adamw_clip_step_gathered": (_c.c_int, [_vp, _vp, _vp, _c.c_int32, _vp, _vp, _c.c_int32,
                                            _c.c_double, _c.c_double, _c.c_double, _c.c_double,
                                            _vp, _c.c_int32, _c.c_int32, _vp]),
    "adamw_rank_total": (_c.c_int, [_vp, _c.c_int32, _c.c_double, _c.c_double,
                                    _c.POINTER(_c.c_double), _c.POINTER(_c.c_double),
                                    _c.POINTER(_c.c_float)]),
    "adamw_clip_step_ranks": (_c.c_int, [_vp, _vp, _vp, _c.c_int32, _vp, _vp, _c.c_int32,
                                         _c.c_double, _c.c_double, _c.c_double, _c.c_double,
                                         _vp, _c.c_int32, _c.c_int32, _vp]),
    "adamw_last_tensor_sumsq": (_c.c_int, [_vp, _vp]),
    "adamw_graph_create": (_c.c_int, [_vp, _vp, _vp, _vp, _vp]),
    "adamw_graph_step": (_c.c_int, [_vp, _c.c_int32, _c.c_double, _c.c_double, _c.c_double,
                                    _vp]),
    "adamw_graph_destroy": (_c.c_int, [_vp]),
    "adamw_record_events": (_c.c_int, [_vp, _vp, _vp, _vp]),
    "adamw_set_launch_options": (_c.c_int, [_vp, _c.c_int32]),
    "adamw_set_decay_mask": (_c.c_int, [_vp, _vp, _c.c_int32]),
    "adamw_clip_step_noalloc": (_c.c_int, [_vp, _vp, _vp, _vp, _c.c_int64, _c.c_int32,
                                           _c.c_double, _c.c_double, _c.c_double,
                                           _c.c_double, _c.c_double, _c.c_double, _vp, _vp]),
    "ckpt_pack": (_c.c_int, [_vp, _c.c_int32, _vp, _vp, _vp, _vp, _vp]),
    "ckpt_write": (_c.c_int, [_vp, _c.c_char_p, _c.c_char_p, _c.c_size_t]),
    "ckpt_write_async": (_c.c_int, [_vp, _c.c_char_p]),
    "ckpt_wait": (_c.c_int, [_vp, _c.c_char_p, _c.c_size_t]),
    "ckpt_set_options": (_c.c_int, [_vp, _c.c_int32, _c.c_int32]),
    "ckpt_step_end": (_c.c_int, [_vp, _c.c_int32, _vp, _vp, _vp, _vp, _vp, _c.c_char_p,
                                 _c.c_int32, _c.POINTER(_c.c_int32)]),
    "ckpt_signals_install": (_c.c_int, [_c.c_int32]),
    "ckpt_signals_take": (_c.c_int32, []),
    "ckpt_write_image": (_c.c_int, [_c.c_char_p, _vp, _c.c_int64, _c.c_int64, _c.c_int32,
                                    _c.c_char_p, _c.c_size_t]),
    "ckpt_rotate": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.POINTER(_c.c_int32)]),
    "ckpt_read": (_c.c_int, [_vp, _c.c_char_p, _c.POINTER(_c.c_int32), _vp, _vp, _vp, _vp]),
    "ckpt_file_size": (_c.c_int64, [_c.c_int64]),
    "ckpt_write_host": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.c_int32, _vp, _vp, _vp,
                                   _c.c_char_p, _c.c_size_t]),
    "ckpt_probe": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.POINTER(_c.c_int32),
                              _c.POINTER(_c.c_int32)]),
    "ckpt_shard_write": (_c.c_int, [_vp, _c.c_char_p, _c.c_int32, _c.c_char_p]),
    "ckpt_shard_write_host": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.c_int32, _c.c_int32, _vp,
                                         _vp, _vp, _c.c_char_p]),
    "ckpt_manifest_commit": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.c_int32, _c.c_double, _vp,
                                        _vp, _c.c_char_p, _c.c_char_p, _c.c_size_t]),
    "ckpt_manifest_load": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.c_int32,
                                      _c.POINTER(_c.c_int32), _c.POINTER(_c.c_int32), _vp, _vp,
                                      _c.c_int32]),
    "ckpt_shard_read": (_c.c_int, [_vp, _c.c_char_p, _c.c_int32, _c.c_int32,
                                   _c.POINTER(_c.c_int32), _vp, _vp, _vp, _vp]),
    "ckpt_consolidate": (_c.c_int, [_c.c_char_p, _c.c_int32, _c.c_char_p, _c.c_char_p,
                                    _c.c_size_t]),
    "ckpt_read_range": (_c.c_int, [_vp, _c.c_char_p, _c.c_int64, _c.POINTER(_c.c_int32), _vp,
                                   _vp, _vp, _vp]),
    "ckpt_sha256_hex": (_c.c_int, [_vp, _c.c_int64, _c.c_char_p]),
    "ckpt_sha256_backend": (_c.c_int, []),
    "adamw_strerror": (_c.c_char_p, [_c.c_int]),
    "adamw_last_error": (_c.c_char_p, []),
}


class LibraryNotBuilt(RuntimeError):
    pass


class AdamWError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {_strerror(status)}: {detail}")
        self.status = status


class NonFiniteGradient(AdamWError):
    """The gradient norm was inf or nan; the update was skipped."""


_lock = threading.Lock()
_lib = None


def library(path: str = None) -> ctypes.CDLL:
    """The loaded C library (loaded once, on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIBRARY
            if not os.path.exists(p):
                raise LibraryNotBuilt(
                    f"{p} is missing: build it with optimizer_step_resumable_gb300.build.build()")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
        return _lib


def _strerror(status: int) -> str:
    return library().adamw_strerror(status).decode()


def _check(status: int, where: str):
    if status != OK:
        detail = library().adamw_last_error().decode()
        cls = NonFiniteGradient if status == ENONFINITE else AdamWError
        raise cls(status, where, detail)


def _stream(stream):
    """cudaStream_t of a torch stream (None: torch's current stream)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _same_device(t, name: str, ctx) -> None:
    if ctx is not None and ctx.device is not None:
        d = t.get_device()
        if d != ctx.device:
            raise ValueError(f"{name} is on cuda:{d}, the context on cuda:{ctx.device}")


def _dev_ptr(t, n: int, name: str, ctx=None) -> int:
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")
    if t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} elements, context has {n}")
    _same_device(t, name, ctx)
    return t.data_ptr()


class Context:
    """Owner of one ``adamw_ctx*``; freed by ``adamw_destroy`` or on GC."""

    def __init__(self, handle: int, n: int, device=None):
        self.handle = handle
        self.n = n
        self.device = device  # CUDA device index the context was created on

    @property
    def num_tensors(self) -> int:
        return library().adamw_num_tensors(self.handle)

    def close(self):
        if self.handle:
            library().adamw_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def adamw_create(n_params: int, offsets=None, numels=None, flags: int = 0) -> Context:
    lib = library()
    if offsets is None and numels is None:
        nt, po, pn, keep = 0, None, None, ()
    else:
        nt = len(offsets)
        if len(numels) != nt:
            raise ValueError("offsets and numels differ in length")
        po = (ctypes.c_int64 * nt)(*offsets)
        pn = (ctypes.c_int64 * nt)(*numels)
        keep = (po, pn)
    out = ctypes.c_void_p()
    st = lib.adamw_create(int(n_params), po and ctypes.addressof(po),
                          pn and ctypes.addressof(pn), nt, int(flags), ctypes.byref(out))
    del keep
    _check(st, "adamw_create")
    import torch
    return Context(out.value, int(n_params), torch.cuda.current_device())


def adamw_destroy(ctx: Context):
    ctx.close()


def adamw_set_hparams(ctx: Context, beta1: float, beta2: float, eps: float):
    _check(library().adamw_set_hparams(ctx.handle, beta1, beta2, eps), "adamw_set_hparams")


def grad_global_norm(ctx: Context, g, wait: bool = True, stream=None):
    """||g||_2; with wait=False returns None and leaves it in the context."""
    out = ctypes.c_double()
    st = library().grad_global_norm(ctx.handle, _dev_ptr(g, ctx.n, "g", ctx),
                                    ctypes.byref(out) if wait else None, _stream(stream))
    _check(st, "grad_global_norm")
    return out.value if wait else None


def adamw_clip_step(ctx: Context, w, g, m, v, t: int, lr: float, wd: float,
                    clip: float, stream=None):
    n = ctx.n
    st = library().adamw_clip_step(ctx.handle, _dev_ptr(w, n, "w", ctx), _dev_ptr(g, n, "g", ctx),
                                   _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx), int(t),
                                   float(lr), float(wd), float(clip), _stream(stream))
    _check(st, "adamw_clip_step")


def adamw_clip_step_ex(ctx: Context, w, g, m, v, t: int, lr: float, wd: float, clip: float,
                       grad_scale: float = 1.0, global_sumsq: float = -1.0,
                       zero_grad: bool = False, tensor_norms: bool = False, stream=None):
    """adamw_clip_step with a gradient scale (micro-batch averaging), an
    optional global sum of squares (sharded state), ZERO_GRAD and
    TENSOR_NORMS."""
    n = ctx.n
    flags = (ZERO_GRAD if zero_grad else 0) | (TENSOR_NORMS if tensor_norms else 0)
    st = library().adamw_clip_step_ex(
        ctx.handle, _dev_ptr(w, n, "w", ctx), _dev_ptr(g, n, "g", ctx), _dev_ptr(m, n, "m", ctx),
        _dev_ptr(v, n, "v", ctx), int(t), float(lr), float(wd), float(clip), float(grad_scale),
        float(global_sumsq), flags, _stream(stream))
    _check(st, "adamw_clip_step_ex")


def _dtype_of(t):
    import torch
    table = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}
    if t.dtype not in table:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return table[t.dtype]


def _typed_ptr(t, n: int, name: str, ctx=None) -> int:
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor")
    if t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} elements, context has {n}")
    _same_device(t, name, ctx)
    return t.data_ptr()


def adamw_clip_step_mixed(ctx: Context, w, g, m, v, t: int, lr: float, wd: float, clip: float,
                          w_lp=None, grad_scale: float = 1.0, global_sumsq: float = -1.0,
                          zero_grad: bool = False, tensor_norms: bool = False, stream=None):
    """Float32 master w, m, v; g float32/bfloat16/float16; optional 16-bit
    copy w_lp (bfloat16 or float16 tensor) of the new weights."""
    n = ctx.n
    flags = (ZERO_GRAD if zero_grad else 0) | (TENSOR_NORMS if tensor_norms else 0)
    lp_ptr, lp_dt = None, DTYPE_BF16
    if w_lp is not None:
        lp_ptr, lp_dt = _typed_ptr(w_lp, n, "w_lp", ctx), _dtype_of(w_lp)
        if lp_dt == DTYPE_F32:
            raise TypeError("w_lp must be bfloat16 or float16")
    st = library().adamw_clip_step_mixed(
        ctx.handle, _dev_ptr(w, n, "w", ctx), _typed_ptr(g, n, "g", ctx), _dtype_of(g), _dev_ptr(m, n, "m", ctx),
        _dev_ptr(v, n, "v", ctx), lp_ptr, lp_dt, int(t), float(lr), float(wd), float(clip),
        float(grad_scale), float(global_sumsq), flags, _stream(stream))
    _check(st, "adamw_clip_step_mixed")


def grad_sumsq_typed(ctx: Context, g, stream=None) -> float:
    out = ctypes.c_double()
    st = library().grad_sumsq_typed(ctx.handle, _typed_ptr(g, ctx.n, "g", ctx), _dtype_of(g),
                                    ctypes.byref(out), _stream(stream))
    _check(st, "grad_sumsq_typed")
    return out.value


def _f64_dev_ptr(t, k: int, name: str, ctx=None) -> int:
    import torch
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float64
            and t.is_contiguous() and t.numel() >= k):
        raise ValueError(f"{name} must be a contiguous CUDA float64 tensor of >= {k} values")
    _same_device(t, name, ctx)
    return t.data_ptr()


def grad_sumsq_to(ctx: Context, g, out, stream=None):
    """This shard's sum of g^2 written to the CUDA float64 tensor `out`
    (its first element) on the stream, with no host wait."""
    st = library().grad_sumsq_to(ctx.handle, _typed_ptr(g, ctx.n, "g", ctx), _dtype_of(g),
                                 _f64_dev_ptr(out, 1, "out", ctx), _stream(stream))
    _check(st, "grad_sumsq_to")


def adamw_clip_step_gathered(ctx: Context, w, g, m, v, t: int, lr: float, wd: float,
                             clip: float, rank_sumsq, grad_scale: float = 1.0,
                             zero_grad: bool = False, stream=None):
    """The fused update of this shard with the global norm added up on the
    device, in rank order, from rank_sumsq (CUDA float64, one value per
    rank, e.g. the output of an all-gather)."""
    n = ctx.n
    world = rank_sumsq.numel()
    st = library().adamw_clip_step_gathered(
        ctx.handle, _dev_ptr(w, n, "w", ctx), _typed_ptr(g, n, "g", ctx), _dtype_of(g),
        _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx), int(t), float(lr), float(wd), float(clip),
        float(grad_scale), _f64_dev_ptr(rank_sumsq, world, "rank_sumsq", ctx), int(world),
        ZERO_GRAD if zero_grad else 0, _stream(stream))
    _check(st, "adamw_clip_step_gathered")


def _f64_host_array(values, name: str):
    """The values as a C array of doubles (ctypes; the caller keeps it alive)."""
    vals = [float(x) for x in values]
    if not vals:
        raise ValueError(f"{name} is empty")
    return (_c.c_double * len(vals))(*vals), len(vals)


def adamw_rank_total(rank_sumsq, clip: float, grad_scale: float = 1.0):
    """(sum, norm, clip factor) of the ranks' sums of squares, added in rank
    order by the library (host only).  Raises NonFiniteGradient (with
    .values = (sum, norm, factor)) when the norm is inf or nan."""
    arr, world = _f64_host_array(rank_sumsq, "rank_sumsq")
    s, norm, scale = _c.c_double(), _c.c_double(), _c.c_float()
    st = library().adamw_rank_total(arr, world, float(clip), float(grad_scale), _c.byref(s),
                                    _c.byref(norm), _c.byref(scale))
    if st == ENONFINITE:
        err = NonFiniteGradient(st, "adamw_rank_total", adamw_last_error())
        err.values = (s.value, norm.value, scale.value)
        raise err
    _check(st, "adamw_rank_total")
    return s.value, norm.value, scale.value


def adamw_clip_step_ranks(ctx: Context, w, g, m, v, t: int, lr: float, wd: float, clip: float,
                          rank_sumsq, grad_scale: float = 1.0, zero_grad: bool = False,
                          stream=None):
    """The fused update of this shard with the global norm of the ranks'
    sums of squares (a host sequence, one float per rank in rank order, e.g.
    gathered over gloo), added up by the library."""
    n = ctx.n
    arr, world = _f64_host_array(rank_sumsq, "rank_sumsq")
    st = library().adamw_clip_step_ranks(
        ctx.handle, _dev_ptr(w, n, "w", ctx), _typed_ptr(g, n, "g", ctx), _dtype_of(g),
        _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx), int(t), float(lr), float(wd),
        float(clip), float(grad_scale), arr, world, ZERO_GRAD if zero_grad else 0,
        _stream(stream))
    _check(st, "adamw_clip_step_ranks")


def grad_tensor_sumsq(ctx: Context, g, stream=None):
    """Per-tensor sums of squares (numpy float64, table order); raises
    NonFiniteGradient (with .values set) if the global sum is not finite."""
    import numpy as np
    out = np.empty(ctx.num_tensors, np.float64)
    st = library().grad_tensor_sumsq(ctx.handle, _dev_ptr(g, ctx.n, "g", ctx), out.ctypes.data,
                                     _stream(stream))
    if st == ENONFINITE:
        err = NonFiniteGradient(st, "grad_tensor_sumsq", adamw_last_error())
        err.values = out
        raise err
    _check(st, "grad_tensor_sumsq")
    return out


def adamw_last_tensor_sumsq(ctx: Context):
    import numpy as np
    out = np.empty(ctx.num_tensors, np.float64)
    _check(library().adamw_last_tensor_sumsq(ctx.handle, out.ctypes.data),
           "adamw_last_tensor_sumsq")
    return out


def grad_sumsq(ctx: Context, g, stream=None) -> float:
    """Sum of g^2 over the context's n values (waits); raises NonFiniteGradient."""
    out = ctypes.c_double()
    st = library().grad_sumsq(ctx.handle, _dev_ptr(g, ctx.n, "g", ctx), ctypes.byref(out),
                              _stream(stream))
    _check(st, "grad_sumsq")
    return out.value


def adamw_graph_create(ctx: Context, w, g, m, v):
    n = ctx.n
    _check(library().adamw_graph_create(ctx.handle, _dev_ptr(w, n, "w", ctx), _dev_ptr(g, n, "g", ctx),
                                        _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx)),
           "adamw_graph_create")


def adamw_graph_step(ctx: Context, t: int, lr: float, wd: float, clip: float, stream=None):
    _check(library().adamw_graph_step(ctx.handle, int(t), float(lr), float(wd), float(clip),
                                      _stream(stream)), "adamw_graph_step")


def adamw_graph_destroy(ctx: Context):
    _check(library().adamw_graph_destroy(ctx.handle), "adamw_graph_destroy")


def adamw_last_norm(ctx: Context):
    """(norm, clip factor) of the last reduction; raises NonFiniteGradient."""
    norm, scale = ctypes.c_double(), ctypes.c_float()
    st = library().adamw_last_norm(ctx.handle, ctypes.byref(norm), ctypes.byref(scale))
    _check(st, "adamw_last_norm")
    return norm.value, scale.value


def adamw_clip_step_noalloc(w, g, m, v, t: int, lr: float, wd: float, clip: float,
                            beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                            norm_out=None, stream=None):
    """The clipped-AdamW step without a context, for callers that must not
    allocate GPU memory (see include/adamw_ckpt.h).  norm_out: optional
    float64 CUDA tensor of one element that receives the gradient norm."""
    import types

    import torch
    n = w.numel()
    here = types.SimpleNamespace(device=torch.cuda.current_device())  # the launch device
    np_ = None
    if norm_out is not None:
        np_ = _f64_dev_ptr(norm_out, 1, "norm_out", here)
    st = library().adamw_clip_step_noalloc(
        _dev_ptr(w, n, "w", here), _dev_ptr(g, n, "g", here), _dev_ptr(m, n, "m", here),
        _dev_ptr(v, n, "v", here),
        int(n), int(t), float(lr), float(wd), float(clip), float(beta1), float(beta2),
        float(eps), np_, _stream(stream))
    _check(st, "adamw_clip_step_noalloc")


def adamw_set_launch_options(ctx: Context, flags: int = 0):
    _check(library().adamw_set_launch_options(ctx.handle, int(flags)),
           "adamw_set_launch_options")


def adamw_set_decay_mask(ctx: Context, decay=None):
    """Per-tensor decay flags (a sequence of bools, one per tensor of the
    context's table; False exempts that tensor from weight decay).  None
    restores decay on every parameter."""
    if decay is None:
        _check(library().adamw_set_decay_mask(ctx.handle, None, 0), "adamw_set_decay_mask")
        return
    flags = (_c.c_uint8 * len(decay))(*[1 if f else 0 for f in decay])
    _check(library().adamw_set_decay_mask(ctx.handle, flags, len(decay)),
           "adamw_set_decay_mask")


def adamw_record_events(ctx: Context, ev_begin=None, ev_mid=None, ev_end=None):
    """The next adamw_clip_step records these torch.cuda.Events (already
    recorded once, so that they exist) around its two kernels."""
    h = [e.cuda_event if e is not None else None for e in (ev_begin, ev_mid, ev_end)]
    _check(library().adamw_record_events(ctx.handle, *h), "adamw_record_events")


def ckpt_pack(ctx: Context, step: int, w, m, v, main_stream=None, side_stream=None):
    n = ctx.n
    ms = _stream(main_stream)
    ss = ms if side_stream is None else _stream(side_stream)
    st = library().ckpt_pack(ctx.handle, int(step), _dev_ptr(w, n, "w", ctx), _dev_ptr(m, n, "m", ctx),
                             _dev_ptr(v, n, "v", ctx), ms, ss)
    _check(st, "ckpt_pack")


def ckpt_write(ctx: Context, directory: str) -> str:
    buf = ctypes.create_string_buffer(4200)
    st = library().ckpt_write(ctx.handle, os.fsencode(directory), buf, len(buf))
    _check(st, "ckpt_write")
    return buf.value.decode()


def ckpt_write_async(ctx: Context, directory: str):
    _check(library().ckpt_write_async(ctx.handle, os.fsencode(directory)), "ckpt_write_async")


def ckpt_wait(ctx: Context) -> str:
    """Path of the last asynchronous write ('' if none); raises on failure."""
    buf = ctypes.create_string_buffer(4200)
    _check(library().ckpt_wait(ctx.handle, buf, len(buf)), "ckpt_wait")
    return buf.value.decode()


def ckpt_set_options(ctx: Context, keep: int = 0, flags: int = CKPT_DIRECT):
    _check(library().ckpt_set_options(ctx.handle, int(keep), int(flags)), "ckpt_set_options")


def ckpt_step_end(ctx: Context, step: int, w, m, v, directory: str, every: int,
                  main_stream=None, side_stream=None) -> int:
    """Checkpoint policy at a step boundary; returns a CKPT_ACTION_* value."""
    n = ctx.n
    ms = _stream(main_stream)
    ss = ms if side_stream is None else _stream(side_stream)
    action = ctypes.c_int32(0)
    st = library().ckpt_step_end(ctx.handle, int(step), _dev_ptr(w, n, "w", ctx),
                                 _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx), ms, ss,
                                 os.fsencode(directory), int(every), ctypes.byref(action))
    _check(st, "ckpt_step_end")
    return action.value


def ckpt_signals_install(mask: int = CKPT_REQ_WRITE | CKPT_REQ_EXIT):
    _check(library().ckpt_signals_install(int(mask)), "ckpt_signals_install")


def ckpt_signals_take() -> int:
    return library().ckpt_signals_take()


def ckpt_write_image(directory: str, image, bytes_: int = None, flags: int = CKPT_DIRECT) -> str:
    """Atomic write of a complete host image (numpy uint8 array, header
    included); the array may be longer than the file (padding for O_DIRECT)."""
    import numpy as np
    if not (isinstance(image, np.ndarray) and image.dtype == np.uint8 and image.flags.c_contiguous):
        raise TypeError("image must be a contiguous uint8 numpy array")
    nbytes = image.size if bytes_ is None else int(bytes_)
    buf = ctypes.create_string_buffer(4200)
    st = library().ckpt_write_image(os.fsencode(directory), image.ctypes.data, nbytes,
                                    image.size, int(flags), buf, len(buf))
    _check(st, "ckpt_write_image")
    return buf.value.decode()


def ckpt_rotate(directory: str, keep: int) -> int:
    removed = ctypes.c_int32(0)
    _check(library().ckpt_rotate(os.fsencode(directory), int(keep), ctypes.byref(removed)),
           "ckpt_rotate")
    return removed.value


def ckpt_read(ctx: Context, path: str, w, m, v, stream=None) -> int:
    n = ctx.n
    step = ctypes.c_int32(-1)
    st = library().ckpt_read(ctx.handle, os.fsencode(path), ctypes.byref(step),
                             _dev_ptr(w, n, "w", ctx), _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx),
                             _stream(stream))
    _check(st, "ckpt_read")
    return step.value


def ckpt_file_size(n: int) -> int:
    return library().ckpt_file_size(int(n))


def ckpt_write_host(directory: str, step: int, w, m, v) -> str:
    """Atomic write of host float32 numpy arrays w, m, v."""
    import numpy as np
    arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in (w, m, v)]
    n = arrs[0].size
    if any(a.size != n for a in arrs):
        raise ValueError("w, m, v differ in size")
    buf = ctypes.create_string_buffer(4200)
    st = library().ckpt_write_host(os.fsencode(directory), int(step), int(n),
                                   *[a.ctypes.data for a in arrs], buf, len(buf))
    _check(st, "ckpt_write_host")
    return buf.value.decode()


def ckpt_probe(path: str, n_expected: int = -1):
    """(step, n) of a valid checkpoint file; raises AdamWError otherwise."""
    step, n = ctypes.c_int32(-1), ctypes.c_int32(-1)
    st = library().ckpt_probe(os.fsencode(path), int(n_expected), ctypes.byref(step),
                              ctypes.byref(n))
    _check(st, "ckpt_probe")
    return step.value, n.value


def ckpt_sha256_backend() -> str:
    """Which code computes the library's SHA-256 digests: "libcrypto" (the
    system's OpenSSL 3) or "builtin"."""
    return "libcrypto" if library().ckpt_sha256_backend() == 1 else "builtin"


def ckpt_sha256_hex(data: bytes) -> str:
    buf = ctypes.create_string_buffer(65)
    st = library().ckpt_sha256_hex(ctypes.c_char_p(data), len(data), buf)
    _check(st, "ckpt_sha256_hex")
    return buf.value.decode()


def ckpt_shard_write(ctx: Context, directory: str, rank: int) -> str:
    """Writes the last packed image as rank<rank>.bin; returns its sha256."""
    buf = ctypes.create_string_buffer(65)
    _check(library().ckpt_shard_write(ctx.handle, os.fsencode(directory), int(rank), buf),
           "ckpt_shard_write")
    return buf.value.decode()


def ckpt_shard_write_host(directory: str, step: int, rank: int, w, m, v) -> str:
    import numpy as np
    arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in (w, m, v)]
    n = arrs[0].size
    buf = ctypes.create_string_buffer(65)
    st = library().ckpt_shard_write_host(os.fsencode(directory), int(step), int(rank), int(n),
                                         *[a.ctypes.data for a in arrs], buf)
    _check(st, "ckpt_shard_write_host")
    return buf.value.decode()


def ckpt_manifest_commit(directory: str, step: int, offsets, numels, digests,
                         wall_clock_seconds: float = 0.0) -> str:
    world = len(offsets)
    po = (ctypes.c_int64 * world)(*offsets)
    pn = (ctypes.c_int64 * world)(*numels)
    buf = ctypes.create_string_buffer(4200)
    st = library().ckpt_manifest_commit(os.fsencode(directory), int(step), world,
                                        float(wall_clock_seconds), ctypes.addressof(po),
                                        ctypes.addressof(pn), "".join(digests).encode(), buf,
                                        len(buf))
    _check(st, "ckpt_manifest_commit")
    return buf.value.decode()


def ckpt_manifest_load(step_dir: str, expected_world: int = -1, verify: bool = True):
    """(step, offsets, numels) of a validated sharded checkpoint."""
    lib = library()
    step, world = ctypes.c_int32(-1), ctypes.c_int32(-1)
    # the shard count first (no digests), then the table at its size
    st = lib.ckpt_manifest_load(os.fsencode(step_dir), int(expected_world), 0,
                                ctypes.byref(step), ctypes.byref(world), None, None, 0)
    _check(st, "ckpt_manifest_load")
    cap = max(1, world.value)
    po = (ctypes.c_int64 * cap)()
    pn = (ctypes.c_int64 * cap)()
    st = lib.ckpt_manifest_load(os.fsencode(step_dir), int(expected_world), 1 if verify else 0,
                                ctypes.byref(step), ctypes.byref(world), ctypes.addressof(po),
                                ctypes.addressof(pn), cap)
    _check(st, "ckpt_manifest_load")
    return step.value, list(po[:world.value]), list(pn[:world.value])


def ckpt_shard_read(ctx: Context, step_dir: str, rank: int, w, m, v, expected_world: int = -1,
                    stream=None) -> int:
    n = ctx.n
    step = ctypes.c_int32(-1)
    st = library().ckpt_shard_read(ctx.handle, os.fsencode(step_dir), int(rank),
                                   int(expected_world), ctypes.byref(step), _dev_ptr(w, n, "w", ctx),
                                   _dev_ptr(m, n, "m", ctx), _dev_ptr(v, n, "v", ctx), _stream(stream))
    _check(st, "ckpt_shard_read")
    return step.value


def ckpt_consolidate(step_dir: str, out_dir: str, expected_world: int = -1) -> str:
    """Writes the flat checkpoint of a sharded one (every shard's sha256
    checked on the way) as <out_dir>/step_NNNNNN.bin; returns its path."""
    buf = ctypes.create_string_buffer(4200)
    st = library().ckpt_consolidate(os.fsencode(step_dir), int(expected_world),
                                    os.fsencode(out_dir), buf, len(buf))
    _check(st, "ckpt_consolidate")
    return buf.value.decode()


def ckpt_read_range(ctx: Context, path: str, offset: int, w, m, v, stream=None) -> int:
    """Reads parameters [offset, offset + ctx.n) of a flat checkpoint into
    w, m, v; returns the stored step."""
    n = ctx.n
    step = ctypes.c_int32(-1)
    st = library().ckpt_read_range(ctx.handle, os.fsencode(path), int(offset),
                                   ctypes.byref(step), _dev_ptr(w, n, "w", ctx), _dev_ptr(m, n, "m", ctx),
                                   _dev_ptr(v, n, "v", ctx), _stream(stream))
    _check(st, "ckpt_read_range")
    return step.value


def adamw_strerror(status: int) -> str:
    return _strerror(status)


def adamw_last_error() -> str:
    return library().adamw_last_error().decode()
