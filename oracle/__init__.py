"""CPU oracle for the clipped-AdamW step and the step_NNNNNN.bin checkpoint.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  The product library
(``optimizer_step_resumable_gb300``) never imports, links or runs it, and the
two share no code: the arithmetic lives in ``oracle.c`` (plain C, double
intermediates, no fused multiply-add), restated from

* "Training as a Recoverable State Transition" (aihero.club), sections
  "The Exact Targets of Clipping and AdamW" and "Example 1";
* "Grow a Language Model: Checkpoints" (unhomeschool.com), section "Format";
* "Checkpoint and Sharded Resume" (AI Engineering from Scratch, lesson 80),
  sections "Atomic write" and "Three failure modes".

This module is argument marshalling around that C file, plus ``build()``
which compiles it with gcc.  Every function is pinned by ``tests/test_oracle_*``
against values and closed forms the pages and the mathematics fix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "_oracle.so")

# The pages' AdamW constants ("The Exact Targets of Clipping and AdamW").
BETA1 = 0.9
BETA2 = 0.999
EPS = 1e-8

# Status codes of oracle.c.
OK, EINVAL, EIO, EFORMAT, ESIZE, EMISMATCH, ENONFINITE = range(7)
STATUS_NAMES = {OK: "OK", EINVAL: "EINVAL", EIO: "EIO", EFORMAT: "EFORMAT",
                ESIZE: "ESIZE", EMISMATCH: "EMISMATCH",
                ENONFINITE: "ENONFINITE"}

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall"]


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: oracle status {STATUS_NAMES.get(status, status)}")
        self.status = status


def build(source: str = SOURCE, output: str = LIBRARY, extra=()) -> str:
    """Compile ``source`` into a shared library at ``output`` with gcc."""
    cmd = ["gcc", *CFLAGS, *extra, source, "-o", output + ".part", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(output + ".part", output)
    return output


class _Terms(ctypes.Structure):
    _fields_ = [(k, ctypes.c_double) for k in
                ("g_hat", "m", "v", "m_hat", "v_hat", "w_decayed", "update", "w")]


_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")


class Oracle:
    """ctypes view of one compiled copy of oracle.c (the default one, or a
    copy compiled elsewhere, e.g. by the mutation tests)."""

    def __init__(self, library: str):
        lib = ctypes.CDLL(library)
        c = ctypes
        lib.oracle_sumsq.argtypes = [_f32p, c.c_int64]
        lib.oracle_sumsq.restype = c.c_double
        lib.oracle_global_norm.argtypes = [_f32p, c.c_int64]
        lib.oracle_global_norm.restype = c.c_double
        lib.oracle_tensor_sumsq.argtypes = [_f32p, _i64p, _i64p, c.c_int32,
                                             np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")]
        lib.oracle_tensor_sumsq.restype = None
        lib.oracle_clip_scale.argtypes = [c.c_double, c.c_double]
        lib.oracle_clip_scale.restype = c.c_double
        lib.oracle_adamw_element.argtypes = [
            c.c_double, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_int32, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_double, c.POINTER(_Terms)]
        lib.oracle_adamw_element.restype = None
        lib.oracle_adamw_clip_step.argtypes = [
            _f32p, _f32p, _f32p, _f32p, c.c_int64, c.c_int32, c.c_double,
            c.c_double, c.c_double, c.c_double, c.c_double, c.c_double,
            c.POINTER(c.c_double)]
        lib.oracle_adamw_clip_step.restype = c.c_int
        lib.oracle_adamw_clip_step_scaled.argtypes = [
            _f32p, _f32p, _f32p, _f32p, c.c_int64, c.c_int32, c.c_double,
            c.c_double, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_double, c.POINTER(c.c_double)]
        lib.oracle_adamw_clip_step_scaled.restype = c.c_int
        lib.oracle_decode16.argtypes = [c.c_uint16, c.c_int32]
        lib.oracle_decode16.restype = c.c_double
        lib.oracle_encode16.argtypes = [c.c_float, c.c_int32]
        lib.oracle_encode16.restype = c.c_uint16
        lib.oracle_adamw_clip_step_mixed.argtypes = [
            _f32p, c.c_void_p, c.c_int32, _f32p, _f32p, c.c_void_p, c.c_int32,
            c.c_int64, c.c_int32, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_double, c.c_double, c.c_double, c.POINTER(c.c_double)]
        lib.oracle_adamw_clip_step_mixed.restype = c.c_int
        lib.oracle_adamw_clip_step_masked.argtypes = [
            _f32p, _f32p, _f32p, _f32p, c.c_int64, _i64p, _i64p, c.c_int32, _u8p,
            c.c_int32, c.c_double, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_double, c.POINTER(c.c_double)]
        lib.oracle_adamw_clip_step_masked.restype = c.c_int
        lib.oracle_adamw_update_range.argtypes = [
            _f32p, _f32p, _f32p, _f32p, c.c_int64, c.c_int64, c.c_double, c.c_int32,
            c.c_double, c.c_double, c.c_double, c.c_double, c.c_double]
        lib.oracle_adamw_update_range.restype = c.c_int
        lib.oracle_adamw_at.argtypes = [
            _i64p, c.c_int64, _f32p, _f32p, _f32p, _f32p, c.c_double,
            c.c_int32, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_double, _f32p, _f32p, _f32p]
        lib.oracle_adamw_at.restype = None
        lib.oracle_adamw_terms_at.argtypes = [
            _i64p, c.c_int64, _f32p, _f32p, _f32p, _f32p, c.c_double,
            c.c_int32, c.c_double, c.c_double, c.c_double, c.c_double,
            c.c_double, np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")]
        lib.oracle_adamw_terms_at.restype = None
        lib.oracle_ckpt_size.argtypes = [c.c_int64]
        lib.oracle_ckpt_size.restype = c.c_int64
        lib.oracle_pack.argtypes = [c.c_int32, c.c_int32, _f32p, _f32p, _f32p, _u8p]
        lib.oracle_pack.restype = c.c_int
        lib.oracle_ckpt_write.argtypes = [
            c.c_char_p, c.c_int32, c.c_int32, _f32p, _f32p, _f32p,
            c.c_char_p, c.c_size_t]
        lib.oracle_ckpt_write.restype = c.c_int
        lib.oracle_ckpt_read.argtypes = [
            c.c_char_p, c.c_int32, c.POINTER(c.c_int32), _f32p, _f32p, _f32p]
        lib.oracle_ckpt_read.restype = c.c_int
        self._lib = lib
        self.library = library

    # --- norm and clip ---------------------------------------------------
    def sumsq(self, g: np.ndarray) -> float:
        g = _f32(g)
        return self._lib.oracle_sumsq(g, g.size)

    def global_norm(self, g: np.ndarray) -> float:
        g = _f32(g)
        return self._lib.oracle_global_norm(g, g.size)

    def tensor_sumsq(self, g, offsets, numels) -> np.ndarray:
        """Sum of squares of each tensor of the offset table (double)."""
        g = _f32(g)
        off = np.ascontiguousarray(offsets, dtype=np.int64)
        num = np.ascontiguousarray(numels, dtype=np.int64)
        if off.size != num.size or (off.size and (off.min() < 0 or (off + num).max() > g.size)):
            raise ValueError("offset table outside g")
        out = np.empty(off.size, np.float64)
        self._lib.oracle_tensor_sumsq(g, off, num, off.size, out)
        return out

    def clip_scale(self, norm: float, clip: float) -> float:
        return self._lib.oracle_clip_scale(float(norm), float(clip))

    # --- AdamW -----------------------------------------------------------
    def adamw_element(self, w, g, m, v, s, t, lr, wd, beta1=BETA1,
                      beta2=BETA2, eps=EPS) -> dict:
        """All intermediates of one update in double (no float32 rounding)."""
        r = _Terms()
        self._lib.oracle_adamw_element(float(w), float(g), float(m), float(v),
                                       float(s), int(t), float(lr), float(wd),
                                       float(beta1), float(beta2), float(eps),
                                       ctypes.byref(r))
        return {k: getattr(r, k) for k, _ in _Terms._fields_}

    def adamw_clip_step(self, w, g, m, v, t, lr, wd, clip, beta1=BETA1,
                        beta2=BETA2, eps=EPS, raise_on_error=True):
        """In-place step over float32 arrays w, m, v; returns (status, norm)."""
        for a in (w, m, v):
            _check_inplace(a)
        g = _f32(g)
        n = w.size
        if not (g.size == m.size == v.size == n):
            raise ValueError("w, g, m, v must have the same size")
        norm = ctypes.c_double()
        st = self._lib.oracle_adamw_clip_step(
            w, g, m, v, n, int(t), float(lr), float(wd), float(clip),
            float(beta1), float(beta2), float(eps), ctypes.byref(norm))
        if st not in (OK, ENONFINITE) or (st != OK and raise_on_error):
            raise OracleError(st, "oracle_adamw_clip_step")
        return st, norm.value

    def adamw_clip_step_scaled(self, w, g, m, v, t, lr, wd, clip, grad_scale,
                               beta1=BETA1, beta2=BETA2, eps=EPS, raise_on_error=True):
        """In-place step on grad_scale * g (gradient accumulation)."""
        for a in (w, m, v):
            _check_inplace(a)
        g = _f32(g)
        norm = ctypes.c_double()
        st = self._lib.oracle_adamw_clip_step_scaled(
            w, g, m, v, w.size, int(t), float(lr), float(wd), float(clip),
            float(grad_scale), float(beta1), float(beta2), float(eps),
            ctypes.byref(norm))
        if st not in (OK, ENONFINITE) or (st != OK and raise_on_error):
            raise OracleError(st, "oracle_adamw_clip_step_scaled")
        return st, norm.value

    # 16-bit formats: dtype 0 = float32, 1 = bfloat16, 2 = IEEE binary16
    def adamw_update_range(self, w, g, m, v, lo, hi, s, t, lr, wd, beta1=BETA1, beta2=BETA2,
                           eps=EPS):
        """In-place update of elements [lo, hi) with the given clip factor s
        (of the whole gradient).  The C call releases the GIL, so threads can
        run disjoint ranges at once."""
        for a in (w, m, v):
            _check_inplace(a)
        g = _f32(g)
        if not (0 <= lo <= hi <= w.size) or not (g.size == m.size == v.size == w.size):
            raise ValueError("range outside the arrays")
        st = self._lib.oracle_adamw_update_range(w, g, m, v, int(lo), int(hi), float(s), int(t),
                                                 float(lr), float(wd), float(beta1),
                                                 float(beta2), float(eps))
        if st != OK:
            raise OracleError(st, "oracle_adamw_update_range")

    def adamw_clip_step_masked(self, w, g, m, v, offsets, numels, decay, t, lr, wd, clip,
                               beta1=BETA1, beta2=BETA2, eps=EPS, raise_on_error=True):
        """In-place step with a per-tensor decay flag (0: that tensor is
        updated with wd = 0); the tensors must tile [0, n) in order."""
        for a in (w, m, v):
            _check_inplace(a)
        g = _f32(g)
        off = np.ascontiguousarray(offsets, dtype=np.int64)
        num = np.ascontiguousarray(numels, dtype=np.int64)
        dec = np.ascontiguousarray(np.asarray(decay) != 0, dtype=np.uint8)
        if not (off.size == num.size == dec.size):
            raise ValueError("offsets, numels and decay differ in length")
        norm = ctypes.c_double()
        st = self._lib.oracle_adamw_clip_step_masked(
            w, g, m, v, w.size, off, num, off.size, dec, int(t), float(lr), float(wd),
            float(clip), float(beta1), float(beta2), float(eps), ctypes.byref(norm))
        if st not in (OK, ENONFINITE) or (st != OK and raise_on_error):
            raise OracleError(st, "oracle_adamw_clip_step_masked")
        return st, norm.value

    def decode16(self, h: int, dtype: int) -> float:
        return self._lib.oracle_decode16(int(h), int(dtype))

    def encode16(self, x: float, dtype: int) -> int:
        return self._lib.oracle_encode16(float(x), int(dtype))

    def adamw_clip_step_mixed(self, w, g, g_dtype, m, v, t, lr, wd, clip,
                              grad_scale=1.0, w_lp_dtype=None, beta1=BETA1,
                              beta2=BETA2, eps=EPS, raise_on_error=True):
        """In-place step with g given as float32 (g_dtype 0) or as uint16
        bit patterns (1 = bfloat16, 2 = binary16); returns (status, norm,
        w_lp) where w_lp holds the new weights rounded to w_lp_dtype."""
        for a in (w, m, v):
            _check_inplace(a)
        if g_dtype == 0:
            g = np.ascontiguousarray(g, dtype=np.float32)
        else:
            g = np.ascontiguousarray(g, dtype=np.uint16)
        if g.size != w.size:
            raise ValueError("g size")
        w_lp = None if w_lp_dtype is None else np.empty(w.size, np.uint16)
        norm = ctypes.c_double()
        st = self._lib.oracle_adamw_clip_step_mixed(
            w, g.ctypes.data, int(g_dtype), m, v,
            None if w_lp is None else w_lp.ctypes.data,
            0 if w_lp_dtype is None else int(w_lp_dtype), w.size, int(t), float(lr),
            float(wd), float(clip), float(grad_scale), float(beta1), float(beta2),
            float(eps), ctypes.byref(norm))
        if st not in (OK, ENONFINITE) or (st != OK and raise_on_error):
            raise OracleError(st, "oracle_adamw_clip_step_mixed")
        return st, norm.value, w_lp

    def adamw_at(self, idx, w, g, m, v, s, t, lr, wd, beta1=BETA1,
                 beta2=BETA2, eps=EPS):
        """New (w, m, v) at indices idx, given the clip factor s."""
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        k = idx.size
        outs = [np.empty(k, np.float32) for _ in range(3)]
        self._lib.oracle_adamw_at(idx, k, _f32(w), _f32(g), _f32(m), _f32(v),
                                  float(s), int(t), float(lr), float(wd),
                                  float(beta1), float(beta2), float(eps),
                                  *outs)
        return tuple(outs)

    TERMS = ("g_hat", "m", "v", "m_hat", "v_hat", "w_decayed", "update", "w")

    def adamw_terms_at(self, idx, w, g, m, v, s, t, lr, wd, beta1=BETA1,
                       beta2=BETA2, eps=EPS) -> np.ndarray:
        """(k, 8) double terms at indices idx, columns as in TERMS."""
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty((idx.size, 8), np.float64)
        self._lib.oracle_adamw_terms_at(idx, idx.size, _f32(w), _f32(g), _f32(m),
                                        _f32(v), float(s), int(t), float(lr),
                                        float(wd), float(beta1), float(beta2),
                                        float(eps), out)
        return out

    # --- checkpoint ------------------------------------------------------
    def ckpt_size(self, n: int) -> int:
        return self._lib.oracle_ckpt_size(int(n))

    def pack(self, step, w, m, v) -> np.ndarray:
        n = w.size
        out = np.empty(self.ckpt_size(n), np.uint8)
        st = self._lib.oracle_pack(int(step), int(n), _f32(w), _f32(m), _f32(v), out)
        if st != OK:
            raise OracleError(st, "oracle_pack")
        return out

    def ckpt_write(self, directory, step, w, m, v) -> str:
        buf = ctypes.create_string_buffer(4200)
        st = self._lib.oracle_ckpt_write(os.fsencode(directory), int(step),
                                         int(w.size), _f32(w), _f32(m), _f32(v),
                                         buf, len(buf))
        if st != OK:
            raise OracleError(st, "oracle_ckpt_write")
        return buf.value.decode()

    def ckpt_read(self, path, n):
        """Returns (status, step, w, m, v); arrays are None unless OK."""
        w = np.empty(n, np.float32)
        m = np.empty(n, np.float32)
        v = np.empty(n, np.float32)
        step = ctypes.c_int32(-1)
        st = self._lib.oracle_ckpt_read(os.fsencode(path), int(n),
                                        ctypes.byref(step), w, m, v)
        if st != OK:
            return st, None, None, None, None
        return st, step.value, w, m, v


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _check_inplace(a):
    if not (isinstance(a, np.ndarray) and a.dtype == np.float32
            and a.flags.c_contiguous and a.flags.writeable):
        raise TypeError("state arrays must be writable contiguous float32")


_lock = threading.Lock()
_default = None


def _stale() -> bool:
    return (not os.path.exists(LIBRARY)
            or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))


def load() -> Oracle:
    """The default oracle, compiled from oracle.c if missing or stale."""
    global _default
    with _lock:
        if _default is None:
            if _stale():
                build()
            _default = Oracle(LIBRARY)
        return _default
